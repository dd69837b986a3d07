// plan.cu -- routing plan: top-k expert ids -> grouped-contiguous layout.
//
// Follows MoonEP PR #38 ("fit planning block size to device SMEM limit"):
// a planning kernel with a per-expert histogram and a per-warp count table
// in shared memory (its scratch is (E+1) x (warps+1) counts), whose block
// size is the largest multiple of one warp whose shared memory fits the
// device's per-block opt-in limit.  The layout itself is the grouped-
// contiguous one of humming PR #129 ("perf(sm90): size grouped W4A8 tiles
// per expert", first section): each expert's rows form one range.
//
// Up to 6144 routed rows (and E small enough for a 32-warp count table) the
// whole plan is ONE block of 1024 threads (plan_small): each warp keeps its
// contiguous sub-chunk of ids in registers, counts it, and after one scan
// places it.  Larger inputs take two launches:
//   plan_hist:    block b counts the ids of its chunk per expert
//                 (warp-aggregated with __match_any_sync) -> ws[b][e].
//   plan_scatter: every block rebuilds the exclusive scan over (expert,
//                 block) from ws, block 0 writes expert_offsets, then each
//                 warp places its contiguous sub-chunk in order: the rank of
//                 an id inside its warp step is the popcount of equal ids on
//                 lower lanes, so the order inside an expert is ascending
//                 source index (stable).
#include "hg_internal.cuh"

namespace hg {
namespace {

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__global__ void plan_hist_kernel(const int32_t* __restrict__ ids, int R, int E, int chunk,
                                 int32_t* __restrict__ ws, uint32_t* status) {
    extern __shared__ int32_t sm_hist[];
    int32_t* cnt = sm_hist;   // [E]
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int begin = blockIdx.x * chunk;
    const int end = min(R, begin + chunk);
    uint32_t bad = 0;
    for (int base = begin + (threadIdx.x & ~31); base < end; base += blockDim.x) {
        const int i = base + lane;
        int key = -2;   // padding lane
        if (i < end) {
            const int e = __ldg(ids + i);
            key = (e >= 0 && e < E) ? e : -1;
        }
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key);
        if (key >= 0 && lane == __ffs(peers) - 1) atomicAdd(&cnt[key], __popc(peers));
        if (key == -1) ++bad;
    }
    if (bad) {
        atomicAdd(&status[kStatusBadIds], bad);
        record_error(status, HG_ERR_BAD_IDS, 0u);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) ws[static_cast<size_t>(blockIdx.x) * E + e] = cnt[e];
}

// Shared memory: per-warp table wc[nw][E], then tot[E] and base[E].
__global__ void plan_scatter_kernel(const int32_t* __restrict__ ids, int R, int E, int chunk,
                                    int nblk, const int32_t* __restrict__ ws,
                                    int32_t* __restrict__ offsets,
                                    int32_t* __restrict__ sorted_to_src,
                                    int32_t* __restrict__ src_to_sorted) {
    extern __shared__ int32_t sm_scat[];
    const int nw = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int32_t* wc = sm_scat;                         // [nw][E]
    int32_t* tot = wc + static_cast<size_t>(nw) * E;
    int32_t* base = tot + E;
    __shared__ int32_t s_total;

    for (int i = threadIdx.x; i < (nw + 2) * E; i += blockDim.x) sm_scat[i] = 0;
    __syncthreads();

    // Totals per expert, and the counts of the blocks before this one.
    const int b = blockIdx.x;
    for (int idx = threadIdx.x; idx < nblk * E; idx += blockDim.x) {
        const int bb = idx / E;
        const int e = idx - bb * E;
        const int v = __ldg(ws + idx);
        if (v) {
            atomicAdd(&tot[e], v);
            if (bb < b) atomicAdd(&base[e], v);
        }
    }
    // Per-warp counts of this block's sub-chunks.
    const int begin = b * chunk;
    const int end = min(R, begin + chunk);
    const int sub = chunk / nw;                    // multiple of 32
    const int wbeg = begin + warp * sub;
    const int wend = min(end, wbeg + sub);
    int32_t* mycnt = wc + static_cast<size_t>(warp) * E;
    for (int s0 = wbeg; s0 < wend; s0 += 32) {
        const int i = s0 + lane;
        int key = -2;
        if (i < wend) {
            const int e = __ldg(ids + i);
            key = (e >= 0 && e < E) ? e : -1;
        }
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key);
        if (key >= 0 && lane == __ffs(peers) - 1) mycnt[key] += __popc(peers);
    }
    __syncthreads();

    // Exclusive scan of the totals over experts (one warp, 32 at a time):
    // off[e]; this block's start for expert e is off[e] + base[e].
    if (warp == 0) {
        int carry = 0;
        for (int c = 0; c < E; c += 32) {
            const int e = c + lane;
            const int v = e < E ? tot[e] : 0;
            int incl = v;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += y;
            }
            if (e < E) {
                const int off = carry + incl - v;
                if (b == 0) offsets[e] = off;
                base[e] += off;
            }
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) {
            s_total = carry;
            if (b == 0) offsets[E] = carry;
        }
    }
    __syncthreads();
    // Per-warp starting rows: base[e] + counts of the earlier warps.
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = base[e];
        for (int w = 0; w < nw; ++w) {
            const int c = wc[static_cast<size_t>(w) * E + e];
            wc[static_cast<size_t>(w) * E + e] = run;
            run += c;
        }
    }
    __syncthreads();

    // Stable placement, warp by warp, step by step in source order.
    const uint32_t lt = lanemask_lt();
    for (int s0 = wbeg; s0 < wend; s0 += 32) {
        const int i = s0 + lane;
        int key = -2;
        if (i < wend) {
            const int e = __ldg(ids + i);
            key = (e >= 0 && e < E) ? e : -1;
        }
        const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key);
        int dest = -1;
        if (key >= 0) dest = mycnt[key] + __popc(peers & lt);
        __syncwarp();
        if (key >= 0 && lane == __ffs(peers) - 1) mycnt[key] += __popc(peers);
        __syncwarp();
        if (i < wend) {
            src_to_sorted[i] = dest;
            if (dest >= 0) sorted_to_src[dest] = i;
        }
    }
    // Rows past the last placed one (only when ids were dropped).
    const int total = s_total;
    for (int j = total + b * blockDim.x + threadIdx.x; j < R; j += nblk * blockDim.x) {
        sorted_to_src[j] = -1;
    }
}


#ifndef HG_PLAN_SMALL_MAX_R
#define HG_PLAN_SMALL_MAX_R 6144
#endif
constexpr int kSmallThreads = 1024;
constexpr int kSmallIdsPerLane = 16;
constexpr int kSmallMaxR = HG_PLAN_SMALL_MAX_R;
static_assert(kSmallMaxR <= kSmallThreads * kSmallIdsPerLane, "ids must fit the registers");

// Shared memory: per-warp table wc[32][E], base[E], then the permutation
// sorted_to_src itself (R entries): placing rows in shared memory and writing
// the array out once, coalesced, avoids R scattered 4-byte global stores
// from a single SM.
__global__ void __launch_bounds__(kSmallThreads)
plan_small_kernel(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ offsets,
                  int32_t* __restrict__ sorted_to_src, int32_t* __restrict__ src_to_sorted,
                  uint32_t* status) {
    extern __shared__ int32_t sm_small[];
    constexpr int nw = kSmallThreads / 32;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int32_t* wc = sm_small;                        // [nw][E]
    int32_t* base = wc + nw * E;                   // [E]
    int32_t* s2d = base + E;                       // [R]
    __shared__ int32_t s_total;

    // Contiguous sub-chunk per warp, a multiple of 32 ids long.
    const int sub = ((R + nw - 1) / nw + 31) & ~31;
    const int wbeg = warp * sub;
    const int wend = min(R, wbeg + sub);
    int key[kSmallIdsPerLane];
#pragma unroll
    for (int j = 0; j < kSmallIdsPerLane; ++j) {
        const int i = wbeg + 32 * j + lane;
        key[j] = -2;
        if (32 * j < sub && i < wend) {
            const int e = __ldg(ids + i);
            key[j] = (e >= 0 && e < E) ? e : -1;
        }
    }
    for (int i = threadIdx.x; i < (nw + 1) * E; i += kSmallThreads) sm_small[i] = 0;
    __syncthreads();

    int32_t* mycnt = wc + warp * E;
    uint32_t bad = 0;
#pragma unroll
    for (int j = 0; j < kSmallIdsPerLane; ++j) {
        if (32 * j < sub) {
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key[j]);
            if (key[j] >= 0 && lane == __ffs(peers) - 1) mycnt[key[j]] += __popc(peers);
            if (key[j] == -1) ++bad;
        }
    }
    if (bad) {
        atomicAdd(&status[kStatusBadIds], bad);
        record_error(status, HG_ERR_BAD_IDS, 0u);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kSmallThreads) {
        int t = 0;
        for (int w = 0; w < nw; ++w) t += wc[w * E + e];
        base[e] = t;
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int c = 0; c < E; c += 32) {
            const int e = c + lane;
            const int v = e < E ? base[e] : 0;
            int incl = v;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += y;
            }
            if (e < E) {
                offsets[e] = carry + incl - v;
                base[e] = carry + incl - v;
            }
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) {
            offsets[E] = carry;
            s_total = carry;
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kSmallThreads) {
        int run = base[e];
        for (int w = 0; w < nw; ++w) {
            const int c = wc[w * E + e];
            wc[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int j = 0; j < kSmallIdsPerLane; ++j) {
        if (32 * j < sub) {
            const int i = wbeg + 32 * j + lane;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key[j]);
            int dest = -1;
            if (key[j] >= 0) dest = mycnt[key[j]] + __popc(peers & lt);
            __syncwarp();
            if (key[j] >= 0 && lane == __ffs(peers) - 1) mycnt[key[j]] += __popc(peers);
            __syncwarp();
            if (i < wend) {
                src_to_sorted[i] = dest;
                if (dest >= 0) s2d[dest] = i;
            }
        }
    }
    __syncthreads();
    const int total = s_total;
    for (int j = threadIdx.x; j < R; j += kSmallThreads) sorted_to_src[j] = j < total ? s2d[j] : -1;
}

}  // namespace

size_t plan_small_smem_bytes(int32_t R, int32_t E) {
    return (static_cast<size_t>(kSmallThreads / 32 + 1) * static_cast<size_t>(E) +
            static_cast<size_t>(R)) * sizeof(int32_t);
}

bool plan_small_fits(int32_t R, int32_t E, int smem_limit) {
    return R <= kSmallMaxR && plan_small_smem_bytes(R, E) <= static_cast<size_t>(smem_limit);
}

size_t plan_smem_bytes(int32_t E, int threads) {
    return static_cast<size_t>(threads / 32 + 2) * static_cast<size_t>(E) * sizeof(int32_t);
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream) {
    if (a.small) {
        const size_t smem = plan_small_smem_bytes(a.R, a.E);
        if (smem > 48 * 1024) {
            cudaError_t err = cudaFuncSetAttribute(plan_small_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
            if (err != cudaSuccess) return err;
        }
        plan_small_kernel<<<1, kSmallThreads, smem, stream>>>(a.ids, a.R, a.E, a.offsets,
                                                               a.sorted_to_src, a.src_to_sorted,
                                                               a.status);
        return cudaGetLastError();
    }
    const size_t smem_hist = static_cast<size_t>(a.E) * sizeof(int32_t);
    const size_t smem_scat = plan_smem_bytes(a.E, a.threads);
    if (smem_scat > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(plan_scatter_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem_scat));
        if (err != cudaSuccess) return err;
    }
    if (smem_hist > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(plan_hist_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem_hist));
        if (err != cudaSuccess) return err;
    }
    plan_hist_kernel<<<a.nblk, a.threads, smem_hist, stream>>>(a.ids, a.R, a.E, a.chunk,
                                                               a.ws_counts, a.status);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    plan_scatter_kernel<<<a.nblk, a.threads, smem_scat, stream>>>(
        a.ids, a.R, a.E, a.chunk, a.nblk, a.ws_counts, a.offsets, a.sorted_to_src,
        a.src_to_sorted);
    return cudaGetLastError();
}

}  // namespace hg
