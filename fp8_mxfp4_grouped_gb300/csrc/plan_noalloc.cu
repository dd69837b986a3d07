// plan_noalloc.cu -- the routing plan for callers that cannot allocate device
// memory.
//
// hg_plan_expert_offsets needs a device workspace for its two-launch path
// (more than 32768 routed rows, or many experts): one count per block per
// expert.  Some callers cannot provide one, because they cannot call
// cudaMalloc at the point where they plan: a host framework that owns every
// device allocation through its own memory pool and does not let a library
// allocate behind its back, or a latency-critical loop that cannot take the
// device-wide synchronisation cudaMalloc and cudaFree may imply.
// hg_plan_expert_offsets_noalloc serves them: its workspace is a fixed-size
// array in this library's device memory.
#include <mutex>

#include "hg_internal.cuh"

namespace hg {
namespace {

// Largest workspace the plan may need here: 65536 counts (256 KiB).  Every
// GPU that loads the library holds this array until the process exits.
constexpr size_t kNoallocScratchInts = 65536;
static __device__ __align__(256) int32_t g_plan_scratch[kNoallocScratchInts];

constexpr int kMaxDevices = 64;
int32_t* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_plan_scratch on the current device.  The first call on
// a device looks it up (cudaGetSymbolAddress, with that device current); in
// host code the array's name is only a host-side stand-in, never a device
// address, so kernels must be given this pointer instead.
hg_status scratch_for_current_device(int32_t** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return HG_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return HG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess) return HG_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_ptr[dev];
    return HG_OK;
}

}  // namespace

void plan_noalloc_reset() {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    for (int d = 0; d < kMaxDevices; ++d) g_scratch_ptr[d] = nullptr;
}

}  // namespace hg

extern "C" hg_status hg_plan_expert_offsets_noalloc(const int32_t* topk_ids, int32_t M,
                                                    int32_t top_k, int32_t E,
                                                    int32_t* expert_offsets,
                                                    int32_t* sorted_to_src,
                                                    int32_t* src_to_sorted, hg_stream_t stream) {
    if (M < 0 || top_k < 1 || E < 1) return HG_ERR_INVALID_ARG;
    const size_t need = hg_plan_workspace_bytes(M, top_k, E);
    if (need == 0) return HG_ERR_UNSUPPORTED_SHAPE;
    if (need > hg::kNoallocScratchInts * sizeof(int32_t)) return HG_ERR_RESOURCE;
    int32_t* scratch = nullptr;
    const hg_status st = hg::scratch_for_current_device(&scratch);
    if (st != HG_OK) return st;
    // The workspace holds per-block counts that the histogram launch writes
    // in full on every call, so nothing in it has to start at zero.
    return hg_plan_expert_offsets(topk_ids, M, top_k, E, expert_offsets, sorted_to_src,
                                  src_to_sorted, scratch, need, stream);
}
