// api.cu -- the extern "C" entry points of libhg (declared in include/hg.h):
// argument validation (before any CUDA call), the plan launch configuration
// (shared-memory fit), TMA tensor-map encoding, and the device status word.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "hg_internal.cuh"

namespace hg {
namespace {

// Library-owned status word; one instance per device (module-scope device
// variable), addressed through cudaGetSymbolAddress.
__device__ uint32_t g_status[kStatusWords];

constexpr int kMaxDevices = 64;
constexpr int kPlanMaxThreads = 512;
constexpr int kPlanIdsPerBlock = 2048;
constexpr int kPlanMaxBlocks = 256;

struct DeviceInfo {
    bool ready = false;
    int num_sms = 0;
    int smem_optin = 0;
    uint32_t* status = nullptr;
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

std::atomic<uint64_t> g_timeout_ns{1000000000ull};
std::atomic<int> g_forced_variant{0};

int choose_variant(int32_t E, int32_t N, int32_t K, int32_t rows, int num_sms) {
    int v = g_forced_variant.load();
    if (!v) v = gemm_pick_variant(E, N, K, rows, num_sms);
    if (v == 4 && N % 256 != 0) v = 8;   // CTA pairs split 256 weight rows
    return v;
}

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;


hg_status device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HG_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return HG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return HG_ERR_CUDA;
        if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
            return HG_ERR_CUDA;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return HG_ERR_CUDA;
        d.status = static_cast<uint32_t*>(p);
        d.ready = true;
    }
    *out = &d;
    return HG_OK;
}

hg_status encoder(PFN_cuTensorMapEncodeTiled_v12000* fn) {
    std::call_once(g_encode_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        }
    });
    if (!g_encode) return HG_ERR_CUDA;
    *fn = g_encode;
    return HG_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Tensor-map cache.  A tensor map depends only on its base address and
// shape, so one encoded for (pointer, sizes) stays valid for any allocation
// at that address with those sizes; the last few of each kind are kept so
// that repeated calls on resident buffers skip the five encodes.
constexpr int kMapCacheEntries = 16;
struct WMapEntry {
    const void* p = nullptr;
    int32_t E = 0, N = 0, K = 0;
    CUtensorMap map;
};
struct AMapEntry {
    const void* p = nullptr;
    int32_t rows = 0, K = 0;
    AMaps maps;
};
struct OMapEntry {
    const void* p = nullptr;
    int32_t rows = 0, N = 0;
    CUtensorMap map;
};
WMapEntry g_wmap[kMapCacheEntries];
AMapEntry g_amap[kMapCacheEntries];
OMapEntry g_omap[kMapCacheEntries];
int g_wmap_next = 0;
int g_amap_next = 0;
int g_omap_next = 0;
std::mutex g_map_mu;

void map_cache_reset() {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < kMapCacheEntries; ++i) {
        g_wmap[i].p = nullptr;
        g_amap[i].p = nullptr;
        g_omap[i].p = nullptr;
    }
    g_wmap_next = g_amap_next = g_omap_next = 0;
}

// Weights: [E*N rows, K elements] of E2M1, unpacked by the TMA into one
// 16-byte chunk (8 data bytes + 8 pad) per 16 elements, 128-byte swizzle,
// boxes of 128 x 128.
hg_status weight_map(PFN_cuTensorMapEncodeTiled_v12000 encode, const uint8_t* w_fp4, int32_t E,
                     int32_t N, int32_t K, CUtensorMap* out) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < kMapCacheEntries; ++i) {
        const WMapEntry& c = g_wmap[i];
        if (c.p == w_fp4 && c.E == E && c.N == N && c.K == K) {
            *out = c.map;
            return HG_OK;
        }
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(K),
                          static_cast<cuuint64_t>(E) * static_cast<cuuint64_t>(N)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(K / 2)};
    cuuint32_t box[2] = {128, 128};
    cuuint32_t estr[2] = {1, 1};
    if (encode(out, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<uint8_t*>(w_fp4), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return HG_ERR_CUDA;
    WMapEntry& slot = g_wmap[g_wmap_next];
    g_wmap_next = (g_wmap_next + 1) % kMapCacheEntries;
    slot.p = w_fp4;
    slot.E = E;
    slot.N = N;
    slot.K = K;
    slot.map = *out;
    return HG_OK;
}

// Activations: [rows, K] bytes, 128-byte swizzle; boxes of 16, 32, 64 and
// 128 rows of 128 bytes.
hg_status act_maps(PFN_cuTensorMapEncodeTiled_v12000 encode, const uint8_t* a_fp8, int32_t rows,
                   int32_t K, AMaps* out) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < kMapCacheEntries; ++i) {
        const AMapEntry& c = g_amap[i];
        if (c.p == a_fp8 && c.rows == rows && c.K == K) {
            *out = c.maps;
            return HG_OK;
        }
    }
    for (int which = 0; which < 4; ++which) {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
        cuuint64_t strides[1] = {static_cast<cuuint64_t>(K)};
        cuuint32_t box[2] = {128, 16u << which};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&out->box[which], CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a_fp8),
                   dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return HG_ERR_CUDA;
    }
    AMapEntry& slot = g_amap[g_amap_next];
    g_amap_next = (g_amap_next + 1) % kMapCacheEntries;
    slot.p = a_fp8;
    slot.rows = rows;
    slot.K = K;
    slot.maps = *out;
    return HG_OK;
}

int plan_nblk(long long R) {
    long long n = (R + kPlanIdsPerBlock - 1) / kPlanIdsPerBlock;
    if (n < 1) n = 1;
    if (n > kPlanMaxBlocks) n = kPlanMaxBlocks;
    return static_cast<int>(n);
}

// Output: [rows, N] BF16 (as 16-bit words), no swizzle, boxes of 16 rows x
// 32 columns, for the epilogues that write whole 16-row chunks with TMA
// stores.
hg_status out_map(PFN_cuTensorMapEncodeTiled_v12000 encode, uint16_t* out, int32_t rows,
                  int32_t N, CUtensorMap* map) {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < kMapCacheEntries; ++i) {
        const OMapEntry& c = g_omap[i];
        if (c.p == out && c.rows == rows && c.N == N) {
            *map = c.map;
            return HG_OK;
        }
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(N) * 2};
    cuuint32_t box[2] = {32, 16};
    cuuint32_t estr[2] = {1, 1};
    if (encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, out, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return HG_ERR_CUDA;
    OMapEntry& slot = g_omap[g_omap_next];
    g_omap_next = (g_omap_next + 1) % kMapCacheEntries;
    slot.p = out;
    slot.rows = rows;
    slot.N = N;
    slot.map = *map;
    return HG_OK;
}

}  // namespace
}  // namespace hg

using namespace hg;

extern "C" {

const char* hg_status_string(int status) {
    switch (status) {
        case HG_OK: return "ok";
        case HG_ERR_INVALID_ARG: return "invalid argument";
        case HG_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case HG_ERR_RESOURCE: return "resource limit exceeded";
        case HG_ERR_CUDA: return "CUDA error";
        case HG_ERR_TIMEOUT: return "device wait timed out";
        case HG_ERR_BAD_OFFSETS: return "expert offsets not monotone or beyond rows";
        case HG_ERR_BAD_IDS: return "expert id out of range";
        default: return "unknown status";
    }
}

int hg_version(void) { return 100; }

hg_status hg_shutdown(void) {
    {
        std::lock_guard<std::mutex> lock(g_dev_mu);
        for (int d = 0; d < kMaxDevices; ++d) g_dev[d] = DeviceInfo{};
    }
    gemm_reset_caches();
    plan_noalloc_reset();
    map_cache_reset();
    return HG_OK;
}

size_t hg_plan_workspace_bytes(int32_t M, int32_t top_k, int32_t E) {
    if (M < 0 || top_k < 1 || E < 1) return 0;
    const long long R = static_cast<long long>(M) * top_k;
    if (R > 0x7FFFFFFFll) return 0;
    return static_cast<size_t>(plan_nblk(R)) * static_cast<size_t>(E) * sizeof(int32_t);
}

int32_t hg_plan_block_threads(int32_t E, int32_t smem_limit_bytes) {
    if (E < 1 || smem_limit_bytes <= 0) return 0;
    for (int t = kPlanMaxThreads; t >= 32; t -= 32) {
        if (plan_smem_bytes(E, t) <= static_cast<size_t>(smem_limit_bytes)) return t;
    }
    return 0;
}

int32_t hg_plan_launches(int32_t M, int32_t top_k, int32_t E) {
    if (M < 0 || top_k < 1 || E < 1) return -1;
    const long long R = static_cast<long long>(M) * top_k;
    if (R > 0x7FFFFFFFll) return -1;
    if (R == 0) return 0;
    DeviceInfo* d = nullptr;
    if (device_info(&d) != HG_OK) return -1;
    if (plan_cluster_ctas(static_cast<int32_t>(R), E, d->smem_optin) > 0) return 1;
    return hg_plan_block_threads(E, d->smem_optin) > 0 ? 2 : -1;
}

hg_status hg_plan_expert_offsets(const int32_t* topk_ids, int32_t M, int32_t top_k, int32_t E,
                                 int32_t* expert_offsets, int32_t* sorted_to_src,
                                 int32_t* src_to_sorted, void* workspace, size_t workspace_bytes,
                                 hg_stream_t stream) {
    if (M < 0 || top_k < 1 || E < 1) return HG_ERR_INVALID_ARG;
    const long long R = static_cast<long long>(M) * top_k;
    if (R > 0x7FFFFFFFll) return HG_ERR_UNSUPPORTED_SHAPE;
    if (!expert_offsets) return HG_ERR_INVALID_ARG;
    if (R > 0 && (!topk_ids || !sorted_to_src || !src_to_sorted)) return HG_ERR_INVALID_ARG;
    const size_t need = hg_plan_workspace_bytes(M, top_k, E);
    if (R > 0 && (!workspace || workspace_bytes < need)) return HG_ERR_INVALID_ARG;
    if (R > 0 && !aligned(workspace, 4)) return HG_ERR_INVALID_ARG;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (R == 0) {
        return cudaMemsetAsync(expert_offsets, 0, sizeof(int32_t) * (E + 1), s) == cudaSuccess
                   ? HG_OK
                   : HG_ERR_CUDA;
    }
    DeviceInfo* d = nullptr;
    hg_status st = device_info(&d);
    if (st != HG_OK) return st;
    const int threads = hg_plan_block_threads(E, d->smem_optin);
    if (threads == 0) return HG_ERR_RESOURCE;
    const int nblk = plan_nblk(R);
    const int step = threads;   // chunk is a multiple of 32 ids per warp
    long long chunk = (R + nblk - 1) / nblk;
    chunk = ((chunk + step - 1) / step) * step;
    PlanArgs a;
    a.ids = topk_ids;
    a.R = static_cast<int32_t>(R);
    a.E = E;
    a.offsets = expert_offsets;
    a.sorted_to_src = sorted_to_src;
    a.src_to_sorted = src_to_sorted;
    a.ws_counts = static_cast<int32_t*>(workspace);
    a.status = d->status;
    a.threads = threads;
    a.nblk = nblk;
    a.chunk = static_cast<int>(chunk);
    a.cluster_ctas = plan_cluster_ctas(a.R, E, d->smem_optin);
    return launch_plan(a, s) == cudaSuccess ? HG_OK : HG_ERR_CUDA;
}

}  // extern "C"

namespace {

hg_status grouped_gemm(const uint8_t* a_fp8, const uint8_t* a_scale, bool a_scale_mmajor,
                       const uint8_t* w_fp4, const uint8_t* w_scale,
                       const int32_t* expert_offsets, int32_t E, int32_t N, int32_t K,
                       int32_t rows, uint16_t* out_bf16, hg_stream_t stream) {
    if (E < 1 || N < 1 || K < 1 || rows < 0) return HG_ERR_INVALID_ARG;
    if (!w_fp4 || !w_scale || !expert_offsets) return HG_ERR_INVALID_ARG;
    if (rows > 0 && (!a_fp8 || !a_scale || !out_bf16)) return HG_ERR_INVALID_ARG;
    if (E > gemm_max_experts() || N % 128 != 0 || K % 128 != 0) return HG_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<long long>(E) * N > 0x7FFFFFFFll) return HG_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(w_fp4, 32) || !aligned(w_scale, 4)) return HG_ERR_INVALID_ARG;
    if (rows > 0 && (!aligned(a_fp8, 16) || !aligned(out_bf16, 2))) return HG_ERR_INVALID_ARG;
    if (rows == 0) return HG_OK;

    DeviceInfo* d = nullptr;
    hg_status st = device_info(&d);
    if (st != HG_OK) return st;
    const int variant = choose_variant(E, N, K, rows, d->num_sms);
    if (static_cast<int>(gemm_smem_bytes(variant, E)) > d->smem_optin) return HG_ERR_RESOURCE;
    PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    st = encoder(&encode);
    if (st != HG_OK) return st;

    CUtensorMap map_w;
    AMaps map_a;
    st = weight_map(encode, w_fp4, E, N, K, &map_w);
    if (st != HG_OK) return st;
    st = act_maps(encode, a_fp8, rows, K, &map_a);
    if (st != HG_OK) return st;
    GemmArgs a;
    a.a_fp8 = a_fp8;
    a.a_scale = a_scale;
    a.w_fp4 = w_fp4;
    a.w_scale = w_scale;
    a.offsets = expert_offsets;
    a.E = E;
    a.N = N;
    a.K = K;
    a.rows = rows;
    a.as_rs = a_scale_mmajor ? 1 : K / 128;
    a.as_ks = a_scale_mmajor ? rows : 1;
    a.out = out_bf16;
    a.status = d->status;
    a.timeout_ns = g_timeout_ns.load();
    a.num_sms = d->num_sms;
    a.variant = variant;
    // The CTA-pair kernel writes whole 16-row chunks of its output tile with
    // TMA stores when the output is 16-byte aligned (the tensor map's base
    // address rule); ragged chunks and unaligned outputs use plain stores.
    CUtensorMap map_o;
    const CUtensorMap* map_o_ptr = nullptr;
    if (variant == 4 && aligned(out_bf16, 16)) {
        st = out_map(encode, out_bf16, rows, N, &map_o);
        if (st != HG_OK) return st;
        map_o_ptr = &map_o;
    }
    return launch_grouped_gemm(a, map_w, map_a, map_o_ptr, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? HG_OK
               : HG_ERR_CUDA;
}

}  // namespace

extern "C" {

hg_status hg_grouped_w4a8_gemm(const uint8_t* a_fp8, const uint8_t* a_scale,
                               const uint8_t* w_fp4, const uint8_t* w_scale,
                               const int32_t* expert_offsets, int32_t E, int32_t N, int32_t K,
                               int32_t rows, uint16_t* out_bf16, hg_stream_t stream) {
    return grouped_gemm(a_fp8, a_scale, false, w_fp4, w_scale, expert_offsets, E, N, K, rows,
                        out_bf16, stream);
}

hg_status hg_grouped_w4a8_gemm_mmajor(const uint8_t* a_fp8, const uint8_t* a_scale_mmajor,
                                      const uint8_t* w_fp4, const uint8_t* w_scale,
                                      const int32_t* expert_offsets, int32_t E, int32_t N,
                                      int32_t K, int32_t rows, uint16_t* out_bf16,
                                      hg_stream_t stream) {
    return grouped_gemm(a_fp8, a_scale_mmajor, true, w_fp4, w_scale, expert_offsets, E, N, K,
                        rows, out_bf16, stream);
}

hg_status hg_quantize_gather_acts(const uint16_t* x_bf16, int32_t M, int32_t K, int32_t top_k,
                                  const int32_t* sorted_to_src, uint8_t* a_fp8,
                                  uint8_t* a_scale, hg_stream_t stream) {
    if (M < 0 || K < 1 || top_k < 1) return HG_ERR_INVALID_ARG;
    if (K % 128 != 0) return HG_ERR_UNSUPPORTED_SHAPE;
    const long long rows = static_cast<long long>(M) * top_k;
    if (rows > 0x7FFFFFFFll) return HG_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return HG_OK;
    if (!x_bf16 || !sorted_to_src || !a_fp8 || !a_scale) return HG_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(a_fp8, 16)) return HG_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    hg_status st = device_info(&d);
    if (st != HG_OK) return st;
    return launch_quantize_gather(x_bf16, K, top_k, sorted_to_src, static_cast<int>(rows), a_fp8,
                                  a_scale, d->num_sms,
                                  reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HG_OK
               : HG_ERR_CUDA;
}

hg_status hg_quantize_scatter_acts(const uint16_t* x_bf16, int32_t M, int32_t K, int32_t top_k,
                                   const int32_t* src_to_sorted, uint8_t* a_fp8,
                                   uint8_t* a_scale, hg_stream_t stream) {
    if (M < 0 || K < 1 || top_k < 1) return HG_ERR_INVALID_ARG;
    if (K % 128 != 0 || top_k > quantize_scatter_max_top_k()) return HG_ERR_UNSUPPORTED_SHAPE;
    const long long rows = static_cast<long long>(M) * top_k;
    if (rows > 0x7FFFFFFFll) return HG_ERR_UNSUPPORTED_SHAPE;
    if (rows == 0) return HG_OK;
    if (!x_bf16 || !src_to_sorted || !a_fp8 || !a_scale) return HG_ERR_INVALID_ARG;
    if (!aligned(x_bf16, 16) || !aligned(a_fp8, 16)) return HG_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    hg_status st = device_info(&d);
    if (st != HG_OK) return st;
    return launch_quantize_scatter(x_bf16, M, K, top_k, src_to_sorted, static_cast<int>(rows),
                                   a_fp8, a_scale, d->num_sms,
                                   reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HG_OK
               : HG_ERR_CUDA;
}

hg_status hg_combine_topk(const uint16_t* y_bf16, const int32_t* src_to_sorted,
                          const float* topk_weights, int32_t M, int32_t top_k, int32_t N,
                          uint16_t* out_bf16, hg_stream_t stream) {
    if (M < 0 || top_k < 1 || N < 1) return HG_ERR_INVALID_ARG;
    if (N % 8 != 0) return HG_ERR_UNSUPPORTED_SHAPE;
    if (static_cast<long long>(M) * top_k > 0x7FFFFFFFll) return HG_ERR_UNSUPPORTED_SHAPE;
    if (M == 0) return HG_OK;
    if (!y_bf16 || !src_to_sorted || !topk_weights || !out_bf16) return HG_ERR_INVALID_ARG;
    if (!aligned(y_bf16, 16) || !aligned(out_bf16, 16) || !aligned(topk_weights, 4))
        return HG_ERR_INVALID_ARG;
    DeviceInfo* d = nullptr;
    hg_status st = device_info(&d);
    if (st != HG_OK) return st;
    return launch_combine_topk(y_bf16, src_to_sorted, topk_weights, M, top_k, N, out_bf16,
                               d->num_sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? HG_OK
               : HG_ERR_CUDA;
}

hg_status hg_get_device_status(hg_stream_t stream, uint32_t* detail) {
    DeviceInfo* d = nullptr;
    hg_status st = device_info(&d);
    if (st != HG_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return HG_ERR_CUDA;
    uint32_t host[kStatusWords] = {0, 0, 0, 0};
    if (cudaMemcpy(host, d->status, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
        return HG_ERR_CUDA;
    const uint32_t zero[kStatusWords] = {0, 0, 0, 0};
    if (cudaMemcpy(d->status, zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
        return HG_ERR_CUDA;
    if (detail) *detail = host[kStatusCode] == HG_ERR_BAD_IDS ? host[kStatusBadIds] : host[kStatusDetail];
    return static_cast<hg_status>(host[kStatusCode]);
}

hg_status hg_selftest_wait_timeout(uint32_t timeout_us, hg_stream_t stream) {
    DeviceInfo* d = nullptr;
    hg_status st = device_info(&d);
    if (st != HG_OK) return st;
    const uint64_t ns = static_cast<uint64_t>(timeout_us ? timeout_us : 1000u) * 1000ull;
    return launch_selftest_wait(d->status, ns, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? HG_OK
               : HG_ERR_CUDA;
}

int32_t hg_gemm_token_tile(int32_t E, int32_t N, int32_t K, int32_t rows) {
    if (E < 1 || N < 1 || K < 1 || rows < 0) return 0;
    DeviceInfo* d = nullptr;
    const int sms = device_info(&d) == HG_OK ? d->num_sms : 0;
    return gemm_variant_token_tile(choose_variant(E, N, K, rows, sms));
}

int32_t hg_gemm_ctas(int32_t E, int32_t N, int32_t K, int32_t rows) {
    if (E < 1 || E > gemm_max_experts() || N < 128 || N % 128 != 0 || K < 128 || K % 128 != 0 ||
        rows < 0)
        return 0;
    DeviceInfo* d = nullptr;
    if (device_info(&d) != HG_OK) return -1;
    GemmArgs a{};
    a.E = E;
    a.N = N;
    a.K = K;
    a.rows = rows;
    a.num_sms = d->num_sms;
    a.variant = choose_variant(E, N, K, rows, d->num_sms);
    return static_cast<int32_t>(gemm_launch_ctas(a));
}

int32_t hg_set_gemm_variant(int32_t variant) {
    if (variant != 0 && variant != 1 && variant != 2 && variant != 4 && variant != 6 &&
        variant != 8)
        return -1;
    return g_forced_variant.exchange(variant);
}

void hg_set_wait_timeout_us(uint32_t timeout_us) {
    g_timeout_ns.store(timeout_us ? static_cast<uint64_t>(timeout_us) * 1000ull : 1000000000ull);
}

}  // extern "C"
