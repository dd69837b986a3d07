// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA tensor
// loads (no multicast), L2 cache policies, tcgen05 (TMEM alloc, block-scaled
// MMA, commit, shared->TMEM copy, TMEM loads, fences) and the shared-memory /
// instruction descriptors the tensor core reads.  Written from the PTX ISA
// description of each instruction.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace hg {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lane_id() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%laneid;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

// One non-blocking-ish probe of the phase with the given parity.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// ------------------------------------------------------------- fences ----

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tcgen05.cp, TMA) of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- TMA ---

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 2-D tiled bulk tensor load global -> shared, completion counted in bytes
// on `bar`.  x is the innermost coordinate (elements), y the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// The same load issued for a CTA pair: the data lands in the executing CTA's
// shared memory and the bytes are counted on `cluster_bar`, an mbarrier in
// either CTA of the pair (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x,
                                                 int32_t y, uint32_t cluster_bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar), "l"(policy)
        : "memory");
}

// 2-D tiled bulk tensor store shared -> global of one box at (x, y), tracked
// in this thread's bulk async-group (commit with bulk_commit_group).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(src)
        : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's committed bulk groups still read
// their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's committed bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void sts_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

// Bring the global bytes of one tensor-map box into L2 (no shared memory,
// no completion tracking).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int32_t x, int32_t y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// Bring `bytes` (multiple of 16) of global memory at a 16-byte aligned
// address into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// -------------------------------------------------------------- tcgen05 --

// Whole warp: allocate `ncols` TMEM columns, base address written to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T with per-32-K block scales from TMEM.
// kind::mxf8f6f4, one scale per row / column per 32-K block (scale_vec::1X).
__device__ __forceinline__ void mma_mxf8f6f4_1x(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t sfa_tmem,
                                                uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// Copy 32 rows x 16 bytes from shared memory into TMEM columns
// [col, col+4) of lanes 0-31, replicated into all four lane quadrants.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t s_desc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(s_desc)
                 : "memory");
}

// Each thread of the warp reads 16 consecutive 32-bit columns of its lane.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------- CTA pairs (clusters) --

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}

// Programmatic dependent launch.  launch_dependents: the next kernel of the
// stream, when launched with programmatic stream serialization, may start
// once every CTA of this grid has executed it (or exited).  wait: in such a
// kernel, block until the preceding grid has completed and its memory
// operations are visible; it returns at once in a kernel launched the
// ordinary way.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Whole cluster: arrive (release) and wait (acquire) on the cluster barrier.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
}

// shared::cluster address of the same shared-memory offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

// 32-bit load from the shared memory of a CTA of the cluster (a
// shared::cluster address from mapa_shared).
__device__ __forceinline__ uint32_t ld_shared_cluster_u32(uint32_t cluster_addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
    return v;
}

// Arrive on an mbarrier in another CTA of the cluster (default semantics:
// release at CTA scope).  Asking for cluster scope instead costs the arriving
// thread ~1800 cycles on GB300.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Store 16 bytes into the shared memory of a CTA of the cluster and count
// them against an mbarrier of that same CTA (complete_tx); both operands are
// shared::cluster addresses.  The receiver sees the data once the barrier's
// phase completes, with no fence on either side.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, uint32_t a, uint32_t b,
                                            uint32_t c, uint32_t d, uint32_t cluster_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, "
        "[%5];" ::"r"(cluster_addr),
        "r"(a), "r"(b), "r"(c), "r"(d), "r"(cluster_bar)
        : "memory");
}

// try_wait with acquire at cluster scope: for barriers other CTAs arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// tcgen05 on a CTA pair: both CTAs allocate / free the same TMEM columns;
// one thread of the even CTA issues copies, MMAs and commits for both.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// M = 256 block-scaled MMA over a CTA pair: A rows 0-127 come from the even
// CTA's shared memory and rows 128-255 from the odd CTA's (same offset); B's
// N columns are split in halves the same way.  Each CTA's TMEM receives its
// 128 rows of D and must hold the scales of its own A rows and of all N
// B columns.
__device__ __forceinline__ void mma_mxf8f6f4_1x_pair(uint32_t d_tmem, uint64_t a_desc,
                                                     uint64_t b_desc, uint32_t idesc,
                                                     uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                     uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// Each CTA of the pair copies 32 rows x 16 bytes of its own shared memory
// (same offset) into its own TMEM, replicated into the four lane quadrants.
__device__ __forceinline__ void tc_cp_32x128b_warpx4_pair(uint32_t taddr, uint64_t s_desc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(s_desc)
                 : "memory");
}

// Arrive once on the mbarrier at offset `bar` in every CTA of `cta_mask` when
// all tcgen05 operations this thread issued so far have completed.
__device__ __forceinline__ void tc_commit_pair_multicast(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

// ------------------------------------------ one elected lane of a warp --
// The same tcgen05 operations, issued by the warp's elected lane (elect.sync
// picks the lowest active lane, so always the same thread while the warp
// stays converged).  The whole warp executes the call with identical
// operands; keeping the issuing loop converged lets its address and
// descriptor arithmetic stay warp-uniform.

__device__ __forceinline__ void mma_mxf8f6f4_1x_elect(uint32_t d_tmem, uint64_t a_desc,
                                                      uint64_t b_desc, uint32_t idesc,
                                                      uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                      uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

// One stage of a single-CTA main loop under a single election: the stage's
// weight- and token-scale copies to TMEM, its four K = 32 block-scaled MMAs
// (operands of MMA kk 32 bytes further on: +2 in the descriptors' address
// field) and the commit that releases the stage.  `accumulate` applies to
// the first MMA only (the others always accumulate).
__device__ __forceinline__ void stage_elect(uint32_t d_tmem, uint32_t sfa_tmem, uint64_t sfa_desc,
                                            uint32_t sfb_tmem, uint64_t sfb_desc, uint64_t a_desc,
                                            uint64_t b_desc, uint32_t idesc0, uint32_t idesc1,
                                            uint32_t idesc2, uint32_t idesc3, uint32_t accumulate,
                                            uint32_t empty_bar) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %11, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "add.s64 a1, %5, 2;\n\tadd.s64 a2, %5, 4;\n\tadd.s64 a3, %5, 6;\n\t"
        "add.s64 b1, %6, 2;\n\tadd.s64 b2, %6, 4;\n\tadd.s64 b3, %6, 6;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%1], %2;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%3], %4;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], %5, %6, %7, [%1], [%3], p;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], a1, b1, %8, [%1], [%3], t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], a2, b2, %9, [%1], [%3], t;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], a3, b3, %10, [%1], [%3], t;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%12];\n\t}" ::"r"(
            d_tmem),
        "r"(sfa_tmem), "l"(sfa_desc), "r"(sfb_tmem), "l"(sfb_desc), "l"(a_desc), "l"(b_desc),
        "r"(idesc0), "r"(idesc1), "r"(idesc2), "r"(idesc3), "r"(accumulate), "r"(empty_bar)
        : "memory");
}

__device__ __forceinline__ void tc_commit_elect(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            bar)
        : "memory");
}

__device__ __forceinline__ void tc_cp_32x128b_warpx4_elect(uint32_t taddr, uint64_t s_desc) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
        "l"(s_desc)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_elect(uint32_t dst, const CUtensorMap* map, int32_t x,
                                                  int32_t y, uint32_t bar, uint64_t policy) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair_elect(uint32_t dst, const CUtensorMap* map,
                                                       int32_t x, int32_t y, uint32_t cluster_bar,
                                                       uint64_t policy) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;\n\t}" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cluster_bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void mma_mxf8f6f4_1x_pair_elect(uint32_t d_tmem, uint64_t a_desc,
                                                           uint64_t b_desc, uint32_t idesc,
                                                           uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
}

__device__ __forceinline__ void tc_cp_32x128b_warpx4_pair_elect(uint32_t taddr, uint64_t s_desc) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
        "l"(s_desc)
        : "memory");
}

__device__ __forceinline__ void tc_commit_pair_multicast_elect(uint32_t bar, uint16_t cta_mask) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%0], %1;\n\t}" ::"r"(bar),
        "h"(cta_mask)
        : "memory");
}

// One stage of the CTA-pair main loop, issued under a single election: the
// stage's weight-scale copy to TMEM, its four K = 32 block-scaled MMAs (MMA kk
// reads operands 32 bytes further on: +2 in a descriptor's address field, which
// cannot carry for shared-memory addresses) and the commit that releases the
// stage in both CTAs.  idesc_kk carries the scale-factor ids of MMA kk;
// `accumulate` applies to the first MMA only (the others always accumulate).
__device__ __forceinline__ void pair_stage_elect(uint32_t d_tmem, uint32_t sfa_tmem,
                                                 uint64_t sfa_desc, uint64_t a_desc,
                                                 uint64_t b_desc, uint32_t idesc0, uint32_t idesc1,
                                                 uint32_t idesc2, uint32_t idesc3,
                                                 uint32_t sfb_tmem, uint32_t accumulate,
                                                 uint32_t empty_bar, uint16_t cta_mask) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "add.s64 a1, %3, 2;\n\tadd.s64 a2, %3, 4;\n\tadd.s64 a3, %3, 6;\n\t"
        "add.s64 b1, %4, 2;\n\tadd.s64 b2, %4, 4;\n\tadd.s64 b3, %4, 6;\n\t"
        "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%1], %2;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], %3, %4, %5, [%1], [%9], p;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], a1, b1, %6, [%1], [%9], t;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], a2, b2, %7, [%1], [%9], t;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], a3, b3, %8, [%1], [%9], t;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
        "[%11], %12;\n\t}" ::"r"(d_tmem),
        "r"(sfa_tmem), "l"(sfa_desc), "l"(a_desc), "l"(b_desc), "r"(idesc0), "r"(idesc1),
        "r"(idesc2), "r"(idesc3), "r"(sfb_tmem), "r"(accumulate), "r"(empty_bar), "h"(cta_mask)
        : "memory");
}

// The same without the commit: one 128-K block of a stage that holds
// several (the commit follows with the stage's last block).
__device__ __forceinline__ void pair_kblock_elect(uint32_t d_tmem, uint32_t sfa_tmem,
                                                  uint64_t sfa_desc, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc0, uint32_t idesc1,
                                                  uint32_t idesc2, uint32_t idesc3,
                                                  uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred e, p, t;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 t, 0, 0;\n\t"
        "add.s64 a1, %3, 2;\n\tadd.s64 a2, %3, 4;\n\tadd.s64 a3, %3, 6;\n\t"
        "add.s64 b1, %4, 2;\n\tadd.s64 b2, %4, 4;\n\tadd.s64 b3, %4, 6;\n\t"
        "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%1], %2;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], %3, %4, %5, [%1], [%9], p;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], a1, b1, %6, [%1], [%9], t;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], a2, b2, %7, [%1], [%9], t;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X "
        "[%0], a3, b3, %8, [%1], [%9], t;\n\t}" ::"r"(d_tmem),
        "r"(sfa_tmem), "l"(sfa_desc), "l"(a_desc), "l"(b_desc), "r"(idesc0), "r"(idesc1),
        "r"(idesc2), "r"(idesc3), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_2d_elect(const CUtensorMap* map, int32_t x, int32_t y) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n\t}" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void bulk_prefetch_l2_elect(const void* p, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
        "@e cp.async.bulk.prefetch.L2.global [%0], %1;\n\t}" ::"l"(reinterpret_cast<uint64_t>(p)),
        "r"(bytes)
        : "memory");
}

// --------------------------------------------------------- descriptors ---

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), the fixed version field, and the swizzle mode.
enum : uint32_t { kSwizzleNone = 0, kSwizzle128B = 2 };

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes,
                                              uint32_t sbo_bytes, uint32_t swizzle) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(swizzle & 0x7u) << 61;
    return d;
}

// K-major operand tile stored as rows of 128 bytes with the 128-byte swizzle
// (the layout a TMA load with CU_TENSOR_MAP_SWIZZLE_128B writes): 8-row
// groups are 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
    return smem_desc(saddr, 16, 1024, kSwizzle128B);
}

// Scale-factor block for tcgen05.cp 32x128b: 32 rows of 16 bytes, unswizzled,
// 8-row core matrices 128 bytes apart.
__device__ __forceinline__ uint64_t desc_sf_32x16(uint32_t saddr) {
    return smem_desc(saddr, 0, 128, kSwizzleNone);
}

// Instruction descriptor for kind::mxf8f6f4 with block scaling.
// Matrix formats: 0 = E4M3, 1 = E5M2, 3 = E2M3, 4 = E3M2, 5 = E2M1.
enum : uint32_t { kFmtE4M3 = 0, kFmtE2M1 = 5 };

__device__ __forceinline__ uint32_t idesc_mxf8f6f4(uint32_t a_fmt, uint32_t b_fmt, uint32_t m,
                                                   uint32_t n) {
    uint32_t d = 0;
    d |= (a_fmt & 0x7u) << 7;     // A format
    d |= (b_fmt & 0x7u) << 10;    // B format
    // bits 13/14: no negation; bits 15/16: A and B K-major
    d |= ((n >> 3) & 0x3Fu) << 17;
    d |= 1u << 23;                // scale factors are UE8M0
    d |= ((m >> 4) & 0x1Fu) << 24;
    return d;
}

// Select which byte of each 32-bit TMEM scale cell the MMA reads.
__device__ __forceinline__ uint32_t idesc_with_sf_ids(uint32_t idesc, uint32_t a_id,
                                                      uint32_t b_id) {
    return idesc | ((a_id & 3u) << 29) | ((b_id & 3u) << 4);
}

}  // namespace ptx
}  // namespace hg
