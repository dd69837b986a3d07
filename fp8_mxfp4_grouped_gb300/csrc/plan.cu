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
// Up to 32768 routed rows (and E small enough for a 32-warp count table) the
// whole plan is ONE launch of one thread-block cluster (plan_cluster, up to
// 8 CTAs): each warp keeps its contiguous sub-chunk of ids in registers,
// counts it, the CTAs exchange their per-expert totals through distributed
// shared memory, and each warp places its ids.  Larger inputs take two
// launches:
//   plan_hist:    block b counts the ids of its chunk per expert
//                 (warp-aggregated: the lanes holding equal ids are found
//                 with one ballot per bit of the id) -> ws[b][e].
//   plan_scatter: every block rebuilds the exclusive scan over (expert,
//                 block) from ws, block 0 writes expert_offsets, then each
//                 warp places its contiguous sub-chunk in order: the rank of
//                 an id inside its warp step is the popcount of equal ids on
//                 lower lanes, so the order inside an expert is ascending
//                 source index (stable).
#include "hg_internal.cuh"
#include "ptx.cuh"

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
    const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;
    for (int base = begin + (threadIdx.x & ~31); base < end; base += blockDim.x) {
        const int i = base + lane;
        int key = -2;   // padding lane
        if (i < end) {
            const int e = __ldg(ids + i);
            key = (e >= 0 && e < E) ? e : -1;
        }
        const uint32_t peers = lanes_with_equal_key(key, nbits);
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
    // the GEMM that follows may start its prologue now (it waits for this
    // grid to complete before it reads the offsets)
    ptx::griddep_launch_dependents();
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
    const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;
    for (int s0 = wbeg; s0 < wend; s0 += 32) {
        const int i = s0 + lane;
        int key = -2;
        if (i < wend) {
            const int e = __ldg(ids + i);
            key = (e >= 0 && e < E) ? e : -1;
        }
        const uint32_t peers = lanes_with_equal_key(key, nbits);
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
        const uint32_t peers = lanes_with_equal_key(key, nbits);
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


// ---------------------------------------------------- one cluster --
//
// Up to kClusterMaxR routed rows (and E small enough for the count tables)
// the whole plan is ONE launch: a cluster of up to 8 CTAs of 1024 threads.
// CTA c of the cluster owns a contiguous chunk of the ids, each of its warps
// a contiguous sub-chunk, held in registers (at most kClusterIdsPerLane per
// lane).  Each warp counts its sub-chunk per expert; the lanes holding equal
// ids are found with one warp ballot per bit of the id (plus one for
// validity), and those masks are kept for the placing pass.  Each CTA then
// turns its per-warp counts into per-warp exclusive prefixes and totals;
// after a cluster barrier every CTA reads all CTAs' totals from their shared
// memory, so it knows the expert offsets and how many ids of each expert the
// lower CTAs hold; a second barrier lets the CTAs go on without their totals
// being read any more.  The placing pass gives id i of expert e the row
// off[e] + (ids of e in lower CTAs, lower warps, earlier warp steps and lower
// lanes): ascending source index inside each expert.
constexpr int kClusterThreads = 1024;
constexpr int kClusterWarps = kClusterThreads / 32;
constexpr int kClusterIdsPerLane = 4;
constexpr int kClusterMaxCtas = 8;
constexpr int kClusterIdsPerCta = kClusterThreads * kClusterIdsPerLane;
constexpr int kClusterMaxR = kClusterMaxCtas * kClusterIdsPerCta;

// Shared memory: per-warp count table wc[32][E] (then per-warp exclusive
// prefixes), then the CTA's totals, the cluster totals and the CTA's bases,
// E entries each.
__global__ void __launch_bounds__(kClusterThreads)
plan_cluster_kernel(const int32_t* __restrict__ ids, int R, int E, int32_t* __restrict__ offsets,
                    int32_t* __restrict__ sorted_to_src, int32_t* __restrict__ src_to_sorted,
                    uint32_t* status) {
    // the GEMM that follows may start its prologue now (it waits for this
    // grid to complete before it reads the offsets)
    ptx::griddep_launch_dependents();
    extern __shared__ int32_t sm_cl[];
    constexpr int nw = kClusterWarps;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int crank = static_cast<int>(ptx::cluster_ctarank());
    const int csize = static_cast<int>(ptx::cluster_nctarank());
    int32_t* wc = sm_cl;                 // [nw][E]
    int32_t* cta_cnt = wc + nw * E;      // [E] ids of each expert in this CTA
    int32_t* tot = cta_cnt + E;          // [E] ids of each expert in the cluster
    int32_t* base = tot + E;             // [E] first row of this CTA's ids of each expert
    __shared__ int32_t s_total;
    const int nbits = E > 1 ? 32 - __clz(E - 1) : 0;

    // This CTA's chunk and this warp's sub-chunk, multiples of 32 ids; every
    // CTA computes the same chunk length.
    const int csz = ((R + csize - 1) / csize + 31) & ~31;
    const int cbeg = crank * csz;
    const int cend = min(R, cbeg + csz);
    const int sub = ((csz + nw - 1) / nw + 31) & ~31;
    const int wbeg = cbeg + warp * sub;
    const int wend = min(cend, wbeg + sub);
    int key[kClusterIdsPerLane];
    uint32_t peers[kClusterIdsPerLane];
#pragma unroll
    for (int j = 0; j < kClusterIdsPerLane; ++j) {
        const int i = wbeg + 32 * j + lane;
        key[j] = -2;
        if (32 * j < sub && i < wend) {
            const int e = __ldg(ids + i);
            key[j] = (e >= 0 && e < E) ? e : -1;
        }
    }
    for (int i = threadIdx.x; i < nw * E; i += kClusterThreads) sm_cl[i] = 0;
    __syncthreads();

    int32_t* mycnt = wc + warp * E;
    uint32_t bad = 0;
#pragma unroll
    for (int j = 0; j < kClusterIdsPerLane; ++j) {
        peers[j] = 0;
        if (32 * j < sub) {
            peers[j] = lanes_with_equal_key(key[j], nbits);
            if (key[j] >= 0 && lane == __ffs(peers[j]) - 1) mycnt[key[j]] += __popc(peers[j]);
            if (key[j] == -1) ++bad;
        }
    }
    if (bad) {
        atomicAdd(&status[kStatusBadIds], bad);
        record_error(status, HG_ERR_BAD_IDS, 0u);
    }
    __syncthreads();
    // per-warp exclusive prefixes and the CTA's totals, one expert per thread
    for (int e = threadIdx.x; e < E; e += kClusterThreads) {
        int run = 0;
#pragma unroll 8
        for (int w = 0; w < nw; ++w) {
            const int c = wc[w * E + e];
            wc[w * E + e] = run;
            run += c;
        }
        cta_cnt[e] = run;
    }
    // every CTA's totals are complete and visible to the cluster
    __syncwarp();
    ptx::cluster_sync();
    const uint32_t cnt_saddr = static_cast<uint32_t>(__cvta_generic_to_shared(cta_cnt));
    for (int e = threadIdx.x; e < E; e += kClusterThreads) {
        int lower = 0, all = 0;
        for (int c = 0; c < csize; ++c) {
            const int v = static_cast<int>(ptx::ld_shared_cluster_u32(
                ptx::mapa_shared(cnt_saddr + 4u * static_cast<uint32_t>(e), static_cast<uint32_t>(c))));
            if (c < crank) lower += v;
            all += v;
        }
        base[e] = lower;
        tot[e] = all;
    }
    // no CTA's totals are read after this point: each CTA may go on and exit
    __syncwarp();
    ptx::cluster_sync();
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
                if (crank == 0) offsets[e] = carry + incl - v;
                base[e] += carry + incl - v;
            }
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) {
            if (crank == 0) offsets[E] = carry;
            s_total = carry;
        }
    }
    __syncthreads();
    const uint32_t lt = lanemask_lt();
#pragma unroll
    for (int j = 0; j < kClusterIdsPerLane; ++j) {
        if (32 * j < sub) {
            const int i = wbeg + 32 * j + lane;
            int dest = -1;
            if (key[j] >= 0) dest = base[key[j]] + mycnt[key[j]] + __popc(peers[j] & lt);
            __syncwarp();
            if (key[j] >= 0 && lane == __ffs(peers[j]) - 1) mycnt[key[j]] += __popc(peers[j]);
            __syncwarp();
            if (i < wend) {
                src_to_sorted[i] = dest;
                if (dest >= 0) sorted_to_src[dest] = i;
            }
        }
    }
    // Rows past the last placed one (only when ids were dropped).
    const int total = s_total;
    for (int j = total + crank * kClusterThreads + static_cast<int>(threadIdx.x); j < R;
         j += csize * kClusterThreads) {
        sorted_to_src[j] = -1;
    }
}

}  // namespace

size_t plan_cluster_smem_bytes(int32_t E) {
    return static_cast<size_t>(kClusterWarps + 3) * static_cast<size_t>(E) * sizeof(int32_t);
}

int plan_cluster_ctas(int32_t R, int32_t E, int smem_limit) {
    if (R > kClusterMaxR || plan_cluster_smem_bytes(E) > static_cast<size_t>(smem_limit)) return 0;
    const int n = (R + kClusterIdsPerCta - 1) / kClusterIdsPerCta;
    return n < 1 ? 1 : n;
}

size_t plan_smem_bytes(int32_t E, int threads) {
    return static_cast<size_t>(threads / 32 + 2) * static_cast<size_t>(E) * sizeof(int32_t);
}

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream) {
    if (a.cluster_ctas > 0) {
        const size_t smem = plan_cluster_smem_bytes(a.E);
        if (smem > 48 * 1024) {
            cudaError_t err = cudaFuncSetAttribute(plan_cluster_kernel,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
            if (err != cudaSuccess) return err;
        }
        if (a.cluster_ctas == 1) {
            // one CTA: a plain launch (a cluster of one is implicit)
            plan_cluster_kernel<<<1, kClusterThreads, smem, stream>>>(
                a.ids, a.R, a.E, a.offsets, a.sorted_to_src, a.src_to_sorted, a.status);
            return cudaGetLastError();
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(a.cluster_ctas), 1, 1);
        cfg.blockDim = dim3(kClusterThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(a.cluster_ctas);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, plan_cluster_kernel, a.ids, a.R, a.E, a.offsets,
                                  a.sorted_to_src, a.src_to_sorted, a.status);
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
