// hg_internal.cuh -- declarations shared by the library's translation units:
// the device status word protocol, the bounded barrier wait, and the host
// launchers each kernel file exports to the C-ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/hg.h"
#include "ptx.cuh"

namespace hg {

// Device status word (3 x uint32, library-owned, one per device):
//   [0] first error code recorded since the last read (0 = none)
//   [1] detail of that first error
//   [2] number of expert ids dropped by the plan (out of range)
enum { kStatusCode = 0, kStatusDetail = 1, kStatusBadIds = 2, kStatusWords = 4 };

__device__ __forceinline__ void record_error(uint32_t* status, uint32_t code, uint32_t detail) {
    if (atomicCAS(&status[kStatusCode], 0u, code) == 0u) {
        atomicExch(&status[kStatusDetail], detail);
    }
}

// Where a wait happened, packed into the status detail of a timeout:
// role in bits 24..31, ring slot / buffer in bits 0..23.
enum WaitRole : uint32_t {
    kRoleProducer = 1,
    kRoleScale = 2,
    kRoleMma = 3,
    kRoleEpilogue = 4,
    kRoleTeardown = 5,
    kRoleSelftest = 6,
    kRoleRelay = 7,
};

struct WaitCtx {
    uint32_t* status;             // device status word
    volatile uint32_t* abort;     // shared-memory abort flag of this CTA
    uint64_t timeout_ns;
};

// Wait for the phase of `bar` with parity `parity` to complete.  Gives up
// after ctx.timeout_ns (records HG_ERR_TIMEOUT and raises the CTA's abort
// flag) or as soon as another role of the CTA raised the abort flag.
// Returns true when the phase completed.  kCluster: acquire at cluster scope
// (for barriers that threads of another CTA of the cluster arrive on).
template <bool kCluster = false>
__device__ __forceinline__ bool try_wait_scoped(uint32_t bar, uint32_t parity) {
    return kCluster ? ptx::mbar_try_wait_cluster(bar, parity) : ptx::mbar_try_wait(bar, parity);
}

template <bool kCluster = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtx& ctx,
                                             uint32_t role, uint32_t where) {
    if (try_wait_scoped<kCluster>(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (try_wait_scoped<kCluster>(bar, parity)) return true;
        if (*ctx.abort) return false;
        if ((it & 7u) == 0u && ptx::globaltimer_ns() - t0 > ctx.timeout_ns) {
            *ctx.abort = 1u;
            record_error(ctx.status, HG_ERR_TIMEOUT, (role << 24) | (where & 0xFFFFFFu));
            return false;
        }
    }
}

// ------------------------------------------------- host-side launchers --

struct GemmArgs {
    const uint8_t* a_fp8;
    const uint8_t* a_scale;
    const uint8_t* w_fp4;
    const uint8_t* w_scale;
    const int32_t* offsets;
    int32_t E, N, K, rows;
    int32_t as_rs, as_ks;   // a_scale element (row r, group g) is at r * as_rs + g * as_ks
    uint16_t* out;
    uint32_t* status;
    uint64_t timeout_ns;
    int num_sms;
    int variant;   // 1, 2, 4 (CTA pairs), 6 (split-K), 8: see hg_set_gemm_variant
};

// Lanes of the warp whose key equals this lane's, for keys in [0, 2^nbits)
// and negative keys (all negative keys of the warp share one class here,
// separate from the valid ones).  Every lane of the warp must call it with
// the same nbits.
__device__ __forceinline__ uint32_t lanes_with_equal_key(int key, int nbits) {
    uint32_t m = __ballot_sync(0xFFFFFFFFu, key < 0);
    if (key >= 0) m = ~m;
    for (int b = 0; b < nbits; ++b) {
        const bool bit = (key >> b) & 1;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, bit);
        m &= bit ? bal : ~bal;
    }
    return m;
}

// Activation tensor maps over the same [rows, K] bytes, 128-byte swizzle,
// with boxes of 128 K x (16 << i) rows: any multiple of 16 rows up to 240
// loads in at most four boxes (one TMA instruction each).
struct AMaps {
    CUtensorMap box[4];
};

// map_out: the output [rows, N] BF16 with boxes of 16 rows x 32 columns, for
// kernels that write whole 16-row chunks with TMA stores; nullptr: plain
// stores only.
cudaError_t launch_grouped_gemm(const GemmArgs& a, const CUtensorMap& map_w, const AMaps& map_a,
                                const CUtensorMap* map_out, cudaStream_t stream);
size_t gemm_smem_bytes(int variant, int32_t E);
long long gemm_launch_ctas(const GemmArgs& a);   // CTAs the launch would use
int gemm_max_experts();
// Forget the per-device kernel settings and occupancy answers (hg_shutdown).
void gemm_reset_caches();
// Forget the plan scratch array's per-device addresses (hg_shutdown).
void plan_noalloc_reset();
int gemm_pick_variant(int32_t E, int32_t N, int32_t K, int32_t rows, int num_sms);
int gemm_variant_token_tile(int variant);
int gemm_variant_max_experts(int variant);

struct PlanArgs {
    const int32_t* ids;
    int32_t R, E;
    int32_t* offsets;
    int32_t* sorted_to_src;
    int32_t* src_to_sorted;
    int32_t* ws_counts;
    uint32_t* status;
    int threads;   // block size chosen by the shared-memory fit
    int nblk;      // number of blocks of the histogram / scatter grids
    int chunk;     // ids per block (multiple of 32)
    int cluster_ctas;   // > 0: whole plan in one cluster of this many CTAs (plan_cluster_ctas)
};

cudaError_t launch_plan(const PlanArgs& a, cudaStream_t stream);
size_t plan_smem_bytes(int32_t E, int threads);
// CTAs of the one-cluster plan for R routed rows and E experts (1..8), or 0
// when R or the count tables exceed what one cluster holds.
int plan_cluster_ctas(int32_t R, int32_t E, int smem_limit);

cudaError_t launch_selftest_wait(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream);

cudaError_t launch_quantize_gather(const uint16_t* x, int K, int top_k, const int32_t* s2d,
                                   int rows, uint8_t* a_fp8, uint8_t* a_scale, int num_sms,
                                   cudaStream_t stream);
cudaError_t launch_quantize_scatter(const uint16_t* x, int M, int K, int top_k, const int32_t* d2s,
                                    int rows, uint8_t* a_fp8, uint8_t* a_scale, int num_sms,
                                    cudaStream_t stream);
int quantize_scatter_max_top_k();
cudaError_t launch_combine_topk(const uint16_t* y, const int32_t* d2s, const float* weights,
                                int M, int top_k, int N, uint16_t* out, int num_sms,
                                cudaStream_t stream);

}  // namespace hg
