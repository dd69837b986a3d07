// gemm_host.cu -- the routing plan and the grouped GEMM on host buffers
// (hg_grouped_w4a8_gemm_host, declared in include/hg.h).
//
// Host code only: it validates every argument before any CUDA call, carves
// the caller's device workspace into the device copies the two steps need,
// and enqueues on the caller's stream: the uploads, hg_plan_expert_offsets,
// hg_grouped_w4a8_gemm and the downloads.  Copies are plain cudaMemcpyAsync
// calls, one per buffer.
#include "hg_internal.cuh"

namespace hg {
namespace {

constexpr size_t kRegionAlign = 256;

size_t round_up(size_t x) { return (x + kRegionAlign - 1) / kRegionAlign * kRegionAlign; }

// Byte offsets of the workspace regions; `total` = 0 for rejected sizes.
struct HostLayout {
    size_t ids, offsets, sorted_to_src, src_to_sorted, plan_ws, a, a_scale, out, total;
    size_t plan_ws_bytes;
};

HostLayout host_layout(int32_t M, int32_t top_k, int32_t E, int32_t N, int32_t K) {
    HostLayout L{};
    if (M < 0 || top_k < 1 || E < 1 || N < 1 || K < 128) return L;
    const long long R = static_cast<long long>(M) * top_k;
    if (R > 0x7FFFFFFFll) return L;
    const size_t r = static_cast<size_t>(R);
    size_t at = 0;
    auto take = [&](size_t bytes) {
        const size_t here = at;
        at += round_up(bytes);
        return here;
    };
    L.ids = take(r * sizeof(int32_t));
    L.offsets = take((static_cast<size_t>(E) + 1) * sizeof(int32_t));
    L.sorted_to_src = take(r * sizeof(int32_t));
    L.src_to_sorted = take(r * sizeof(int32_t));
    L.plan_ws_bytes = hg_plan_workspace_bytes(M, top_k, E);
    L.plan_ws = take(L.plan_ws_bytes);
    L.a = take(r * static_cast<size_t>(K));
    L.a_scale = take(r * static_cast<size_t>(K / 128));
    L.out = take(r * static_cast<size_t>(N) * sizeof(uint16_t));
    L.total = at;
    return L;
}

bool is_aligned(const void* p, uintptr_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace
}  // namespace hg

extern "C" {

size_t hg_gemm_host_workspace_bytes(int32_t M, int32_t top_k, int32_t E, int32_t N, int32_t K) {
    return hg::host_layout(M, top_k, E, N, K).total;
}

hg_status hg_grouped_w4a8_gemm_host(const int32_t* topk_ids_host, const uint8_t* a_fp8_host,
                                    const uint8_t* a_scale_host, const uint8_t* w_fp4,
                                    const uint8_t* w_scale, int32_t M, int32_t top_k, int32_t E,
                                    int32_t N, int32_t K, uint16_t* out_bf16_host,
                                    int32_t* expert_offsets_host, int32_t* sorted_to_src_host,
                                    void* workspace, size_t workspace_bytes, hg_stream_t stream) {
    using hg::is_aligned;
    // -- every check the two device calls make, before anything is enqueued
    if (M < 0 || top_k < 1 || E < 1) return HG_ERR_INVALID_ARG;
    const long long R = static_cast<long long>(M) * top_k;
    if (R > 0x7FFFFFFFll) return HG_ERR_UNSUPPORTED_SHAPE;
    if (E > hg::gemm_max_experts() || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0)
        return HG_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<long long>(E) * N > 0x7FFFFFFFll) return HG_ERR_UNSUPPORTED_SHAPE;
    if (!w_fp4 || !w_scale || !is_aligned(w_fp4, 32) || !is_aligned(w_scale, 4))
        return HG_ERR_INVALID_ARG;
    if (R > 0 && (!topk_ids_host || !a_fp8_host || !a_scale_host || !out_bf16_host))
        return HG_ERR_INVALID_ARG;
    const hg::HostLayout L = hg::host_layout(M, top_k, E, N, K);
    if (!workspace || !is_aligned(workspace, hg::kRegionAlign) || workspace_bytes < L.total)
        return HG_ERR_INVALID_ARG;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* ids = reinterpret_cast<int32_t*>(ws + L.ids);
    int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.offsets);
    int32_t* sorted_to_src = reinterpret_cast<int32_t*>(ws + L.sorted_to_src);
    int32_t* src_to_sorted = reinterpret_cast<int32_t*>(ws + L.src_to_sorted);
    uint8_t* a = ws + L.a;
    uint8_t* a_scale = ws + L.a_scale;
    uint16_t* out = reinterpret_cast<uint16_t*>(ws + L.out);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const size_t r = static_cast<size_t>(R);

    if (r > 0) {
        if (cudaMemcpyAsync(ids, topk_ids_host, r * sizeof(int32_t), cudaMemcpyHostToDevice, s) !=
                cudaSuccess ||
            cudaMemcpyAsync(a, a_fp8_host, r * static_cast<size_t>(K), cudaMemcpyHostToDevice,
                            s) != cudaSuccess ||
            cudaMemcpyAsync(a_scale, a_scale_host, r * static_cast<size_t>(K / 128),
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
            return HG_ERR_CUDA;
    }
    hg_status st = hg_plan_expert_offsets(ids, M, top_k, E, offsets, sorted_to_src, src_to_sorted,
                                          ws + L.plan_ws, L.plan_ws_bytes, stream);
    if (st != HG_OK) return st;
    if (r > 0) {
        st = hg_grouped_w4a8_gemm(a, a_scale, w_fp4, w_scale, offsets, E, N, K,
                                  static_cast<int32_t>(R), out, stream);
        if (st != HG_OK) return st;
        if (cudaMemcpyAsync(out_bf16_host, out, r * static_cast<size_t>(N) * sizeof(uint16_t),
                            cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return HG_ERR_CUDA;
        if (sorted_to_src_host &&
            cudaMemcpyAsync(sorted_to_src_host, sorted_to_src, r * sizeof(int32_t),
                            cudaMemcpyDeviceToHost, s) != cudaSuccess)
            return HG_ERR_CUDA;
    }
    if (expert_offsets_host &&
        cudaMemcpyAsync(expert_offsets_host, offsets, (static_cast<size_t>(E) + 1) * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return HG_ERR_CUDA;
    return HG_OK;
}

}  // extern "C"
