// gemm.cu -- grouped-contiguous FP8 E4M3 x MXFP4 E2M1 GEMM on tcgen05.
//
// What is computed follows humming PR #129 ("perf(sm90): size grouped W4A8
// tiles per expert"): benchmark command (float8e4m3 activations with one
// float8e8m0 scale per row per 128-K group, float4e2m1 weights with one
// float8e8m0 scale per output column per 32-K group, bfloat16 output,
// grouped_contiguous rows) and its first section (the tile is sized from the
// rows of each expert, not from the total row count).
//
// Design (GB300 / sm_103a):
//  * swap-AB: the weight rows of one expert (128 per tile) are the MMA's M
//    side, the expert's routed tokens are the MMA's N side.  N can be any
//    multiple of 16 up to 256, so each expert's token tile is sized from its
//    own row count at instruction granularity: an expert with 130 rows gets
//    one 144-token tile, not two 128-row tiles.
//  * persistent CTAs (one or two per SM, sized to one wave) walk a unit list
//    (expert, weight-row tile, token tile) built on the device from
//    expert_offsets; no host sync.  CTA pairs with at most four rounds of
//    units give the largest experts an extra token tile where the last
//    round has room for it.
//  * warp roles: warp 0 issues the TMA loads (weights through the
//    16U4_ALIGN16B unpacking TMA type, activations as bytes in boxes of
//    128/64/32/16 rows; both with the L2 evict-last hint; no multicast);
//    one scale warp per ring slot (2, 3, 8, ...) stages the block scales
//    into the tensor core's scale layout (activation scales are per 128-K,
//    replicated into the four 32-K blocks they cover; the CTA-pair kernel
//    instead packs four 128-K blocks' activation scales into one scale word,
//    staged by a warp of its own, and picks the byte with the MMA's
//    scale-factor id) and arrives on the stage's TMA barrier, so the MMA warp
//    waits on one barrier per stage; warp 1 copies scales to TMEM and issues
//    tcgen05.mma kind::mxf8f6f4 with block scaling (a stage under one
//    election), accumulating FP32 in TMEM; warps 4..7 drain the TMEM
//    accumulator to BF16 with stores cut at the expert's last row (two
//    accumulator buffers, or one where two 224-row pipelines share an SM's
//    TMEM; CTA pairs write whole 16-row chunks with TMA tensor stores).
//  * variants (GemmCfg): token tile, ring depth, CTAs per SM, accumulator
//    buffers; split-K over clusters of four (partials reduce-scattered
//    through distributed shared memory); and a CTA-pair kernel (tcgen05
//    cta_group::2, grouped_w4a8_pair_kernel, stages of 256 K where K
//    allows).  The host picks one from the mean rows per expert
//    (gemm_pick_variant): measured thresholds, and wave models of the
//    resident CTAs for the split-K and single-CTA 224-row variants.
//  * launched with programmatic dependent launch: barrier set-up, TMEM
//    allocation and tensor-map prefetch run while the routing plan's last
//    kernel finishes; griddepcontrol.wait comes before the first read of
//    expert_offsets.
//  * every barrier wait is bounded (see wait_bounded).
#include <cuda_bf16.h>

#include <mutex>

#include "hg_internal.cuh"

namespace hg {
namespace {

constexpr int kBK = 128;              // K per pipeline stage = one activation-scale group
constexpr int kBW = 128;              // weight rows per tile (MMA M)
constexpr int kEpiWarps = 4;
constexpr int kMaxE = 512;            // scheduler tables live in shared memory
constexpr int kPairFillRounds = 4;    // CTA pairs: fill the last round up to this many rounds
static_assert(kMaxE <= 32 * 32, "the last-round fill keeps one bit per expert and lane");
constexpr uint32_t kWTileBytes = kBW * kBK;    // unpacked E2M1: one byte of smem per element
// The 16U4_ALIGN16B TMA load writes 8 data bytes into each 16-byte chunk and
// leaves the other 8 untouched; its transaction count is the packed bytes.
constexpr uint32_t kWTileTx = kBW * kBK / 2;
constexpr uint32_t kSfaBytes = 512;            // 128 rows x 4 blocks of 32 K
constexpr uint32_t kSmemPerSm = 233472;        // 228 KB per SM on sm_103
constexpr uint32_t kSmemPerBlockMax = 232448;  // 227 KB opt-in per block
constexpr uint32_t kSmemReservedPerBlock = 1024;

// One pipeline shape.  T: largest token tile (MMA N); S: ring stages; C: CTAs
// resident per SM.  Each CTA is a complete pipeline; with C = 2 two MMA
// issuers share the SM's tensor core (one thread issues one MMA per ~80-130
// cycles, so small tiles need two issuers to keep up with HBM).
// CL > 1: the grid runs as clusters of CL CTAs, and the kernel may split the
// K loop of every unit over 2 or CL of them (split-K, chosen on the device
// from the unit count); each CTA then holds receive slots for the FP32
// partial tiles of the others.
// AB: TMEM accumulator buffers.  With AB = 1 the MMAs of the next unit wait
// for the epilogue to drain the accumulator (the other CTA on the SM keeps the
// tensor core busy meanwhile); it lets a 224-row token tile run two CTAs per SM.
// SA: the activation boxes of a stage are issued by the stage's scale warp
// instead of the producer (more warps issuing TMA; measured faster for the
// 112-row tiles, slower for the 224-row ones).
template <int T, int S, int C, int CL = 1, int AB = 2, bool SA = false>
struct GemmCfg {
    static constexpr bool kScaleWarpsLoadA = SA;
    static constexpr int kTMax = T;
    static constexpr int kStages = S;
    static constexpr int kCtasPerSm = C;
    static constexpr int kCluster = CL;
    static constexpr int kAccBufs = AB;
    // A CTA of a split group finalises 4/s of the four TMEM lane quadrants
    // and receives s-1 partials of each: (4/s)(s-1) slots, at most 3.
    static constexpr uint32_t kRxSlotBytes = 32 * T * 4;     // one lane quadrant, FP32
    static constexpr int kRxSlots = CL == 1 ? 0 : (CL == 2 ? 2 : 3);
    static constexpr uint32_t kRxBytes = kRxSlots * kRxSlotBytes;
    // scale warps take the stages in turn: one per ring slot.  Each must own
    // exactly one slot: its waits on the slot's empty barrier are parity
    // waits, which are only exact for the phase right after the one it last
    // waited for (a warp visiting a slot several ring revolutions apart could
    // see an older phase of the same parity complete).
    static constexpr int kSfWarps = S;
    static constexpr int kThreads = 32 * (6 + kSfWarps);   // TMA, MMA, 4 epilogue, scale warps
    static constexpr uint32_t kATileBytes = T * kBK;
    static constexpr int kSfbAtoms = T > 128 ? 2 : 1;      // 128 tokens per scale block
    static constexpr uint32_t kSfbBytes = 512 * kSfbAtoms;
    static constexpr uint32_t kAccCols = T;               // TMEM columns per accumulator buffer
    static constexpr uint32_t kTmemCols = 512 / C;
    static constexpr uint32_t kSfCol0 = AB * kAccCols;     // scale slots after the buffers
    static constexpr uint32_t kSfSlotCols = 4 + 4 * kSfbAtoms;
    static constexpr uint32_t kOffW = 0;                   // [stage] weight tiles
    static constexpr uint32_t kOffA = kOffW + S * kWTileBytes;
    static constexpr uint32_t kOffSfa = kOffA + S * kATileBytes;
    static constexpr uint32_t kOffSfb = kOffSfa + S * kSfaBytes;
    static constexpr uint32_t kOffRx = kOffSfb + S * kSfbBytes;
    static constexpr uint32_t kOffBar = kOffRx + kRxBytes;
    static constexpr uint32_t kOffMisc = kOffBar + 256;
    static constexpr uint32_t kOffSched = kOffMisc + 64;
    static constexpr size_t smem_bytes(int E) {
        return kOffSched + static_cast<size_t>(5 * E + 1) * sizeof(int32_t) + 1024;
    }
    static constexpr size_t kSmemBudget =
        C == 1 ? kSmemPerBlockMax : kSmemPerSm / C - kSmemReservedPerBlock;
    static_assert(CL == 1 || CL == 2 || CL == 4, "split over 2 or 4 CTAs");
    static_assert(S <= 4, "scale warps 2, 3, 8, 9: one per ring slot");
    static_assert(AB == 2 || (AB == 1 && CL == 1), "one accumulator buffer, without split-K");
    static_assert(8 * (2 * S + 5 + 8) <= 256, "barrier area");
    // experts whose scheduler tables still fit next to the ring (<= kMaxE)
    static constexpr int kMaxExperts =
        (static_cast<long long>(kSmemBudget) - static_cast<long long>(smem_bytes(0))) / 20 < kMaxE
            ? static_cast<int>((kSmemBudget - smem_bytes(0)) / 20)
            : kMaxE;
    static_assert(T % 16 == 0 && T >= 16 && T <= 240, "MMA N; at most four activation boxes");
    static_assert(kOffA % 1024 == 0 && kATileBytes % 1024 == 0, "swizzle atoms need 1024-B alignment");
    static_assert(kSfCol0 + S * kSfSlotCols <= kTmemCols, "TMEM budget");
    static_assert(kMaxExperts >= 32 && smem_bytes(kMaxExperts) <= kSmemBudget,
                  "shared memory budget");
    static_assert(C * kThreads * 96 <= 65536, "registers for C resident CTAs");
};

// CTA-pair shape (tcgen05 cta_group::2).  T: largest token tile (MMA N,
// multiple of 32, split in halves between the two CTAs); S: ring stages; KB:
// 128-K blocks per stage.  Each CTA holds its 128 weight rows and half of the
// token tile per block, so a pair computes a 256 x T tile with one MMA
// instruction stream.  With KB = 2 the MMA warp waits and commits once per
// eight MMAs instead of four: on CTA pairs the MMA warp's own per-stage work
// bounds the tensor pipe.
// Token scales travel in groups of kSfbGroup 128-K blocks: an activation
// scale covers a whole block, so the four bytes of a TMEM scale word, which
// the MMA selects by its B scale-factor id, can carry four blocks' scales of
// one token instead of one block's scale four times.  One copy to TMEM per
// group then replaces one per block (the per-block token-scale copies of CTA
// pairs measured 6-7 % of the launch at large M on GB300).
template <int T, int S, int C, int KB = 1>
struct PairCfg {
    static constexpr int kTMax = T;
    static constexpr int kHalf = T / 2;
    static constexpr int kStages = S;
    static constexpr int kCtasPerSm = C;
    static constexpr int kKB = KB;
    static constexpr int kSfWarps = S;      // one per ring slot (see GemmCfg)
    static constexpr int kSfbWarp = 6 + S;  // token scales, one group at a time
    static constexpr int kThreads = 32 * (7 + S);
    static constexpr int kSfbGroup = 4;     // 128-K blocks per token-scale group
    static constexpr int kSfbSlots = 3;     // token-scale groups in flight
    static constexpr uint32_t kATileBytes = kHalf * kBK;
    static constexpr uint32_t kWStageBytes = KB * kWTileBytes;
    static constexpr uint32_t kAStageBytes = KB * kATileBytes;
    static constexpr uint32_t kSfaStageBytes = KB * kSfaBytes;
    static constexpr int kSfbAtoms = T > 128 ? 2 : 1;
    static constexpr uint32_t kSfbBytes = 512 * kSfbAtoms;
    static constexpr uint32_t kAccCols = T;
    static constexpr uint32_t kTmemCols = 512 / C;
    static constexpr uint32_t kSfCol0 = 2 * kAccCols;            // weight scales: 4 columns per block
    static constexpr uint32_t kSfbCol0 = kSfCol0 + 4 * KB * S;   // token scales: 4 per atom per group slot
    static constexpr uint32_t kOffW = 0;
    static constexpr uint32_t kOffA = kOffW + S * kWStageBytes;
    static constexpr uint32_t kOffSfa = kOffA + S * kAStageBytes;
    static constexpr uint32_t kOffSfb = kOffSfa + S * kSfaStageBytes;   // [group slot] token scales
    // output staging: per epilogue warp two 16-row x 32-column BF16 buffers
    static constexpr uint32_t kOutChunkBytes = 16 * 32 * 2;
    static constexpr uint32_t kOffOut = kOffSfb + kSfbSlots * kSfbBytes;
    static constexpr uint32_t kOffBar = kOffOut + kEpiWarps * 2 * kOutChunkBytes;
    static constexpr uint32_t kOffMisc = kOffBar + 256;
    static constexpr uint32_t kOffSched = kOffMisc + 64;
    static constexpr size_t smem_bytes(int E) {
        return kOffSched + static_cast<size_t>(5 * E + 1) * sizeof(int32_t) + 1024;
    }
    static constexpr size_t kSmemBudget =
        C == 1 ? kSmemPerBlockMax : kSmemPerSm / C - kSmemReservedPerBlock;
    static_assert(T % 32 == 0 && T >= 32 && T <= 256, "MMA N, split in two halves of 16k");
    static_assert(kOffA % 1024 == 0 && kATileBytes % 1024 == 0, "swizzle atoms need 1024-B alignment");
    static_assert(kSfbCol0 + kSfbSlots * 4 * kSfbAtoms <= kTmemCols, "TMEM budget");
    static_assert(smem_bytes(kMaxE) <= kSmemBudget, "shared memory budget");
    static_assert(8 * (2 * S + 5 + 2 * kSfbSlots) <= 256, "barrier area");
    static_assert(C * kThreads * 96 <= 65536, "registers for C resident CTAs");
    static_assert(kSfbGroup == 4, "four 128-K blocks per 32-bit scale word");
    static_assert(KB == 1 || KB == 2, "a token-scale group is whole stages");
};

using CfgPair = PairCfg<224, 5, 1>;       // many rows per expert, N % 256 == 0
using CfgPair2 = PairCfg<224, 3, 1, 2>;   // the same with 256-K stages, K % 256 == 0

using CfgSmall = GemmCfg<64, 4, 2>;    // few rows per expert: HBM-bound weight streaming
using CfgMid = GemmCfg<112, 3, 2, 1, 2, true>;   // a few hundred rows per expert
using CfgSplit = GemmCfg<32, 4, 2, 4>; // few units per CTA: split-K over clusters of 4
using CfgWide2 = GemmCfg<224, 2, 2, 1, 1>;   // 224-row tiles, two CTAs per SM, one TMEM buffer each

// Split-K factor for a launch of G CTAs (a multiple of max_split) over U
// units of KT stages: the s in {1, 2, 4} dividing KT that minimises the
// stages of the busiest CTA, ceil(U / (G / s)) * KT / s; ties keep the
// smaller split.
__host__ __device__ __forceinline__ int choose_split(int U, int KT, int G, int max_split) {
    int best = 1;
    long long best_cost = static_cast<long long>((U + G - 1) / G) * KT;
    for (int s = 2; s <= max_split; s <<= 1) {
        if (KT % s != 0) continue;
        const int groups = G / s;
        const long long c = static_cast<long long>((U + groups - 1) / groups) * (KT / s);
        if (c < best_cost) {
            best_cost = c;
            best = s;
        }
    }
    return best;
}

struct Sched {
    const int32_t* start;
    const int32_t* rows;
    const int32_t* ntt;
    const int32_t* tile;
    const int32_t* prefix;   // [E+1] exclusive prefix of units per expert
    int E;
    int NT;                  // weight-row tiles per expert (N / (128 * blocks per unit))
    int wstep;               // weight rows per unit (128 * blocks per unit)
};

struct Unit {
    int e;
    int n0;      // first weight row (output column)
    int row0;    // first sorted row of the token tile
    int nrows;   // valid rows of the tile
    int n_mma;   // MMA N: nrows rounded up to 16
};

__device__ __forceinline__ Unit decode_unit(const Sched& s, int u) {
    int lo = 0, hi = s.E;   // prefix[lo] <= u < prefix[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s.prefix[mid] <= u) lo = mid; else hi = mid;
    }
    Unit t;
    t.e = lo;
    const int local = u - s.prefix[lo];
    const int ntt = s.ntt[lo];
    const int nt = local / ntt;
    const int tt = local - nt * ntt;
    const int tile = s.tile[lo];
    t.n0 = nt * s.wstep;
    t.row0 = s.start[lo] + tt * tile;
    t.nrows = min(tile, s.rows[lo] - tt * tile);
    t.n_mma = (t.nrows + 15) & ~15;
    return t;
}

__device__ __forceinline__ uint32_t ldg_u32(const uint8_t* p) {
    return __ldg(reinterpret_cast<const uint32_t*>(p));
}

__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

// Bounded wait that ignores the abort flag: used while draining in-flight
// asynchronous work before the CTA exits.
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer_ns() - t0 > timeout_ns) return false;
    }
    return true;
}

// Load `n` activation rows (a multiple of 16, at most 240) starting at row
// `row`, K offset `k`, into the swizzled tile at `dst`: one TMA per set bit
// of n / 16, largest box first, so a tile takes at most four instructions.
// kPair: the CTA-pair form, `bar` a shared::cluster address in either CTA.
// kElect: called by a whole converged warp, issued by its elected lane.
template <bool kPair = false, bool kElect = false>
__device__ __forceinline__ void load_a_rows(const AMaps& maps, uint32_t dst, int k, int row, int n,
                                            uint32_t bar, uint64_t policy) {
    int r = 0;
#pragma unroll
    for (int i = 3; i >= 0; --i) {
        const int h = 16 << i;
        if (n & h) {
            if (kPair && kElect) {
                ptx::tma_load_2d_pair_elect(dst + r * kBK, &maps.box[i], k, row + r, bar, policy);
            } else if (kPair) {
                ptx::tma_load_2d_pair(dst + r * kBK, &maps.box[i], k, row + r, bar, policy);
            } else if (kElect) {
                ptx::tma_load_2d_elect(dst + r * kBK, &maps.box[i], k, row + r, bar, policy);
            } else {
                ptx::tma_load_2d(dst + r * kBK, &maps.box[i], k, row + r, bar, policy);
            }
            r += h;
        }
    }
}

template <class Cfg>
__global__ void __launch_bounds__(Cfg::kThreads, Cfg::kCtasPerSm)
grouped_w4a8_kernel(const __grid_constant__ CUtensorMap map_w,
                    const __grid_constant__ AMaps map_a,
                    const uint8_t* __restrict__ a_scale, const uint8_t* __restrict__ w_scale,
                    const int32_t* __restrict__ offsets, int E, int N, int K, int rows,
                    int as_rs, int as_ks, uint16_t* __restrict__ out, uint32_t* status,
                    uint64_t timeout_ns) {
    constexpr int kStages = Cfg::kStages;
    constexpr int kTMax = Cfg::kTMax;
    constexpr int kCL = Cfg::kCluster;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (sbase - raw_u32);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // bar_full_tma: a stage's tiles have landed (the producer's expect-tx
    // arrival and the bytes) and its scales are staged (one arrival from the
    // stage's scale warp), so the MMA warp waits on one barrier per stage.
    const uint32_t bar_full_tma = sbase + Cfg::kOffBar;
    const uint32_t bar_empty = bar_full_tma + 8 * kStages;
    const uint32_t bar_tfull = bar_empty + 8 * kStages;
    const uint32_t bar_tempty = bar_tfull + 16;
    const uint32_t bar_done = bar_tempty + 16;
    // split-K: per lane quadrant, "partials received" (arrive + bytes) and
    // "my partial consumed by its owner" (one remote arrive)
    const uint32_t bar_rx_full = bar_done + 8;
    const uint32_t bar_tx_free = bar_rx_full + 32;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(base + Cfg::kOffMisc);
    int32_t* s_start = reinterpret_cast<int32_t*>(base + Cfg::kOffSched);
    int32_t* s_rows = s_start + E;
    int32_t* s_ntt = s_rows + E;
    int32_t* s_tile = s_ntt + E;
    int32_t* s_prefix = s_tile + E;   // E + 1 entries

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar_full_tma + 8 * s, 2);
            ptx::mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_tfull + 8 * b, 1);
            ptx::mbar_init(bar_tempty + 8 * b, kEpiWarps);
        }
        ptx::mbar_init(bar_done, 1);
        if (kCL > 1) {
            for (int q = 0; q < 4; ++q) {
                ptx::mbar_init(bar_rx_full + 8 * q, 1);
                ptx::mbar_init(bar_tx_free + 8 * q, 1);
            }
        }
        misc[1] = 0u;   // abort flag
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(sbase + Cfg::kOffMisc, Cfg::kTmemCols);
        ptx::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&map_w);
        for (int i = 0; i < 4; ++i) ptx::prefetch_tensormap(&map_a.box[i]);
    }

    // Nothing above reads global memory: with programmatic dependent launch
    // it overlaps the kernel before (the routing plan); from here on the
    // kernel reads what that kernel wrote.
    ptx::griddep_wait();

    // Per-expert token tiling, from the expert's own row count.
    const int NT = N / kBW;
    for (int e = threadIdx.x; e < E; e += Cfg::kThreads) {
        const int lo = offsets[e];
        const int hi = offsets[e + 1];
        int r = 0;
        if (lo < 0 || hi < lo || hi > rows) {
            record_error(status, HG_ERR_BAD_OFFSETS, static_cast<uint32_t>(e));
        } else {
            r = hi - lo;
        }
        const int ntt = (r + kTMax - 1) / kTMax;
        const int tile = ntt ? ((((r + ntt - 1) / ntt) + 15) & ~15) : 0;
        s_start[e] = lo;
        s_rows[e] = r;
        s_ntt[e] = ntt;
        s_tile[e] = tile;
        s_prefix[e] = ntt * NT;
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int c = 0; c < E; c += 32) {
            const int e = c + lane;
            const int v = e < E ? s_prefix[e] : 0;
            int incl = v;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += y;
            }
            if (e < E) s_prefix[e] = carry + incl - v;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) s_prefix[E] = carry;
    }
    ptx::tc_fence_before();
    if (kCL > 1) {
        __syncwarp();
        ptx::cluster_sync();   // every CTA's barriers exist before any remote arrive
    } else {
        __syncthreads();
    }
    ptx::tc_fence_after();

    const uint32_t tmem_base = misc[0];
    const Sched sch{s_start, s_rows, s_ntt, s_tile, s_prefix, E, NT, kBW};
    const int U = s_prefix[E];
    const int KT = K / kBK;
    const WaitCtx wctx{status, misc + 1, timeout_ns};
    // Split-K: groups of `split` consecutive CTAs (inside one cluster) share
    // each unit, CTA krank of a group taking stages [k0, k1).  Every CTA
    // derives the same split from U.  Without clusters the loops below read
    // blockIdx / gridDim / 0 / KT directly: holding the group geometry in
    // registers across the warp roles slowed the single MMA-issuing thread
    // by 15-19 % at large M (measured on GB300).
    int split = 1, krank = 0, gid = 0, ngroups = 1, k0 = 0, k1 = KT;
    if constexpr (kCL > 1) {
        split = choose_split(U, KT, static_cast<int>(gridDim.x), kCL);
        krank = static_cast<int>(blockIdx.x) % split;
        gid = static_cast<int>(blockIdx.x) / split;
        ngroups = static_cast<int>(gridDim.x) / split;
        k0 = krank * (KT / split);
        k1 = k0 + KT / split;
    }

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        // Like the MMA issuer: the whole warp walks the loop, the elected
        // lane issues, waits are agreed on with a vote.
        const uint64_t pol_w = ptx::policy_evict_last();   // weight tiles are re-read by the other token tiles of their expert
        const uint64_t pol_a = ptx::policy_evict_last();
        uint32_t g = 0;
        bool ok = true;
        for (int u = kCL > 1 ? gid : static_cast<int>(blockIdx.x); ok && u < U;
             u += kCL > 1 ? ngroups : static_cast<int>(gridDim.x)) {
            const Unit t = decode_unit(sch, u);
            const int wrow = t.e * N + t.n0;
            for (int ks = kCL > 1 ? k0 : 0; ks < (kCL > 1 ? k1 : KT); ++ks, ++g) {
                const uint32_t slot = g % kStages;
                const uint32_t ph = (g / kStages) & 1u;
                if (!__all_sync(0xFFFFFFFFu, wait_bounded(bar_empty + 8 * slot, ph ^ 1u, wctx,
                                                          kRoleProducer, slot))) {
                    ok = false;
                    break;
                }
                const uint32_t fb = bar_full_tma + 8 * slot;
                ptx::mbar_arrive_expect_tx_elect(fb, kWTileTx + t.n_mma * kBK);
                ptx::tma_load_2d_elect(sbase + Cfg::kOffW + slot * kWTileBytes, &map_w, ks * kBK,
                                       wrow, fb, pol_w);
                if constexpr (!Cfg::kScaleWarpsLoadA) {
                    load_a_rows<false, true>(map_a, sbase + Cfg::kOffA + slot * Cfg::kATileBytes,
                                             ks * kBK, t.row0, t.n_mma, fb, pol_a);
                }
            }
        }
        // No copy may land after the CTA exits: wait for the last ring's
        // worth of issued loads (all of them on the normal path already).
        const uint32_t first = g > kStages ? g - kStages : 0;
        for (uint32_t gg = first; gg < g; ++gg) {
            wait_drain(bar_full_tma + 8 * (gg % kStages), (gg / kStages) & 1u, timeout_ns);
        }
    } else if (warp == 1) {
        // ------------------------------------------------- MMA issuer ---
        // The whole warp walks the units and stages with identical values;
        // every tcgen05 instruction is issued by its elected lane.  Waits
        // are polled by every lane and agreed on with a vote, so the warp
        // stays converged and its address and descriptor arithmetic stays
        // warp-uniform.
        uint32_t g = 0, tc = 0;
        bool ok = true;
        for (int u = kCL > 1 ? gid : static_cast<int>(blockIdx.x); ok && u < U;
             u += kCL > 1 ? ngroups : static_cast<int>(gridDim.x), ++tc) {
            const Unit t = decode_unit(sch, u);
            const uint32_t b = tc % Cfg::kAccBufs;
            if (!__all_sync(0xFFFFFFFFu,
                            wait_bounded(bar_tempty + 8 * b, ((tc / Cfg::kAccBufs) & 1u) ^ 1u, wctx,
                                         kRoleMma, 0x100u | b))) {
                break;
            }
            ptx::tc_fence_after();
            const uint32_t idesc0 =
                ptx::idesc_mxf8f6f4(ptx::kFmtE2M1, ptx::kFmtE4M3, kBW, t.n_mma);
            const uint32_t d_tmem = tmem_base + b * Cfg::kAccCols;
            for (int ks = kCL > 1 ? k0 : 0; ks < (kCL > 1 ? k1 : KT); ++ks, ++g) {
                const uint32_t slot = g % kStages;
                const uint32_t ph = (g / kStages) & 1u;
                if (!__all_sync(0xFFFFFFFFu,
                                wait_bounded(bar_full_tma + 8 * slot, ph, wctx, kRoleMma, slot))) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                // scale slot: [weight block: 4 cols][token atoms: 4 cols each]
                const uint32_t sf_col = tmem_base + Cfg::kSfCol0 + slot * Cfg::kSfSlotCols;
                const uint32_t sfb_col = sf_col + 4;
                const uint32_t sfa = sbase + Cfg::kOffSfa + slot * kSfaBytes;
                const uint32_t sfb = sbase + Cfg::kOffSfb + slot * Cfg::kSfbBytes;
                if (Cfg::kSfbAtoms > 1 && t.n_mma > 128) {
                    ptx::tc_cp_32x128b_warpx4_elect(sfb_col + 4, ptx::desc_sf_32x16(sfb + 512));
                }
                const uint32_t wsm = sbase + Cfg::kOffW + slot * kWTileBytes;
                const uint32_t asm_ = sbase + Cfg::kOffA + slot * Cfg::kATileBytes;
                static_assert(kBK / 32 == 4, "four K = 32 MMAs per stage");
                ptx::stage_elect(d_tmem, sf_col, ptx::desc_sf_32x16(sfa), sfb_col,
                                 ptx::desc_sf_32x16(sfb), ptx::desc_kmajor_sw128(wsm),
                                 ptx::desc_kmajor_sw128(asm_), ptx::idesc_with_sf_ids(idesc0, 0, 0),
                                 ptx::idesc_with_sf_ids(idesc0, 1, 1),
                                 ptx::idesc_with_sf_ids(idesc0, 2, 2),
                                 ptx::idesc_with_sf_ids(idesc0, 3, 3),
                                 ks != (kCL > 1 ? k0 : 0) ? 1u : 0u, bar_empty + 8 * slot);
            }
            if (!ok) break;
            ptx::tc_commit_elect(bar_tfull + 8 * b);
        }
        // Everything issued must finish before TMEM is released.
        ptx::tc_commit_elect(bar_done);
        wait_drain(bar_done, 0u, timeout_ns);
    } else if (warp >= 4 && warp < 4 + kEpiWarps) {
        // ---------------------------------------------------- epilogue --
        const int q = warp & 3;   // TMEM lane quadrant this warp may read
        // Split-K reduce-scatter: quadrant q of every unit is finalised by
        // group rank `owner`; the other ranks send it their FP32 partial of
        // that quadrant (st.async into the owner's receive slot), and the
        // owner adds the partials in K order (rank 0 first), so the result
        // does not depend on timing.
        const int owner = (q * split) >> 2;
        const bool finalise = owner == krank;
        const uint32_t rank0 = kCL > 1 ? ptx::cluster_ctarank() - krank : 0;   // group's first CTA
        const int per_owner = 4 / split;                       // quadrants each rank finalises
        const uint32_t rx_base =
            sbase + Cfg::kOffRx + (q - owner * per_owner) * (split - 1) * Cfg::kRxSlotBytes;
        uint32_t tc = 0;
        bool armed = false;   // a receive was announced and not yet seen complete
        for (int u = kCL > 1 ? gid : static_cast<int>(blockIdx.x); u < U;
             u += kCL > 1 ? ngroups : static_cast<int>(gridDim.x), ++tc) {
            const Unit t = decode_unit(sch, u);
            const uint32_t b = tc % Cfg::kAccBufs;
            if (!wait_bounded(bar_tfull + 8 * b, (tc / Cfg::kAccBufs) & 1u, wctx, kRoleEpilogue, b)) break;
            ptx::tc_fence_after();
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * Cfg::kAccCols;
            if constexpr (kCL == 1) {
                const int n = t.n0 + 32 * q + lane;
                uint16_t* dst = out + static_cast<size_t>(t.row0) * N + n;
                for (int c0 = 0; c0 < t.nrows; c0 += 16) {
                    uint32_t v[16];
                    ptx::tmem_ld_32x32b_x16(taddr + c0, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < t.nrows) {
                            dst[static_cast<size_t>(c0 + j) * N] = __bfloat16_as_ushort(
                                __float2bfloat16_rn(__uint_as_float(v[j])));
                        }
                    }
                }
            } else if (!finalise) {
                // ---- send this quadrant's partial to its owner
                if (!wait_bounded<true>(bar_tx_free + 8 * q, (tc & 1u) ^ 1u, wctx, kRoleEpilogue,
                                        0x200u | q)) {
                    break;
                }
                const uint32_t dst_rank = rank0 + owner;
                const int slot = (krank - owner - 1 + split) % split;
                const uint32_t dst =
                    ptx::mapa_shared(rx_base + slot * Cfg::kRxSlotBytes + 16 * lane, dst_rank);
                const uint32_t dbar = ptx::mapa_shared(bar_rx_full + 8 * q, dst_rank);
                for (int c0 = 0; c0 < t.n_mma; c0 += 16) {
                    uint32_t v[16];
                    ptx::tmem_ld_32x32b_x16(taddr + c0, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        // layout [column / 4][lane][column % 4]
                        ptx::st_async_v4(dst + (c0 / 4 + jj) * 512, v[4 * jj], v[4 * jj + 1],
                                         v[4 * jj + 2], v[4 * jj + 3], dbar);
                    }
                }
            } else {
                // ---- finalise: own partial (+ the others' in K order) -> BF16
                if (kCL > 1 && split > 1) {
                    const uint32_t rxb = bar_rx_full + 8 * q;
                    if (lane == 0) {
                        ptx::mbar_arrive_expect_tx(
                            rxb, static_cast<uint32_t>((split - 1) * 32 * t.n_mma * 4));
                    }
                    armed = true;
                    if (!wait_bounded<true>(rxb, tc & 1u, wctx, kRoleEpilogue, 0x300u | q)) break;
                    armed = false;
                }
                const int n = t.n0 + 32 * q + lane;
                uint16_t* dst = out + static_cast<size_t>(t.row0) * N + n;
                const float4* rx = reinterpret_cast<const float4*>(
                    base + (rx_base - sbase)) + lane;
                for (int c0 = 0; c0 < t.nrows; c0 += 16) {
                    uint32_t v[16];
                    ptx::tmem_ld_32x32b_x16(taddr + c0, v);
                    ptx::tmem_ld_wait();
                    float acc[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] = 0.0f;
                    for (int k = 0; k < split; ++k) {
                        if (k == krank) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) acc[j] += __uint_as_float(v[j]);
                        } else {
                            const int slot = (k - krank - 1 + split) % split;
                            const float4* p = rx + slot * (Cfg::kRxSlotBytes / 16) + (c0 / 4) * 32;
#pragma unroll
                            for (int jj = 0; jj < 4; ++jj) {
                                const float4 w = p[jj * 32];
                                acc[4 * jj] += w.x;
                                acc[4 * jj + 1] += w.y;
                                acc[4 * jj + 2] += w.z;
                                acc[4 * jj + 3] += w.w;
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < t.nrows) {
                            dst[static_cast<size_t>(c0 + j) * N] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(acc[j]));
                        }
                    }
                }
                if (kCL > 1 && split > 1) {
                    // slots read: let each sender write its next partial
                    __syncwarp();
                    if (lane == 0) {
                        for (int k = 0; k < split; ++k) {
                            if (k != krank) {
                                ptx::mbar_arrive_remote(
                                    ptx::mapa_shared(bar_tx_free + 8 * q, rank0 + k));
                            }
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar_tempty + 8 * b);
        }
        if (kCL > 1 && armed) {
            // gave up while partials were on their way: let them land first
            wait_drain(bar_rx_full + 8 * q, tc & 1u, timeout_ns);
        }
    } else {
        // ------------------------------------------- scale staging -----
        const int sfw = (warp < 4) ? warp - 2 : warp - 8 + 2;   // warps 2, 3, 8, 9, ...
        const int ws_row = K / 32;     // bytes per w_scale row
        const uint64_t pol_a = ptx::policy_evict_last();
        uint32_t g = 0;
        bool ok = true;
        for (int u = kCL > 1 ? gid : static_cast<int>(blockIdx.x); ok && u < U;
                 u += kCL > 1 ? ngroups : static_cast<int>(gridDim.x)) {
            const Unit t = decode_unit(sch, u);
            const uint8_t* wsrc = w_scale + static_cast<size_t>(t.e * N + t.n0 + lane) * ws_row;
            for (int ks = kCL > 1 ? k0 : 0; ks < (kCL > 1 ? k1 : KT); ++ks, ++g) {
                if (static_cast<int>(g % Cfg::kSfWarps) != sfw) continue;
                const uint32_t slot = g % kStages;
                const uint32_t ph = (g / kStages) & 1u;
                // Weight scales: row n = lane + 32c, the four 32-K blocks of
                // this stage in one 32-bit word (byte i = block i).
                uint32_t wv[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    wv[c] = ldg_u32(wsrc + static_cast<size_t>(32 * c) * ws_row + ks * 4);
                }
                // Token scales: one per 128-K group, replicated into the four
                // 32-K blocks.  Token index = 128a + lane + 32c.
                uint32_t av[4 * Cfg::kSfbAtoms];
#pragma unroll
                for (int i = 0; i < 4 * Cfg::kSfbAtoms; ++i) {
                    const int tok = 128 * (i >> 2) + lane + 32 * (i & 3);
                    const int r = t.row0 + tok;
                    av[i] = 0x7F7F7F7Fu;
                    if (tok < t.n_mma && r < rows) {
                        av[i] = static_cast<uint32_t>(
                                    __ldg(a_scale + static_cast<size_t>(r) * as_rs +
                                          static_cast<size_t>(ks) * as_ks)) *
                                0x01010101u;
                    }
                }
                if (!__all_sync(0xFFFFFFFFu,
                                wait_bounded(bar_empty + 8 * slot, ph ^ 1u, wctx, kRoleScale, slot))) {
                    ok = false;
                    break;
                }
                if constexpr (Cfg::kScaleWarpsLoadA) {
                    // counted on the stage's full barrier, armed by the producer
                    load_a_rows<false, true>(map_a, sbase + Cfg::kOffA + slot * Cfg::kATileBytes,
                                             ks * kBK, t.row0, t.n_mma, bar_full_tma + 8 * slot,
                                             pol_a);
                }
                const uint32_t sfa = sbase + Cfg::kOffSfa + slot * kSfaBytes + 16 * lane;
                const uint32_t sfb = sbase + Cfg::kOffSfb + slot * Cfg::kSfbBytes + 16 * lane;
                sts_v4(sfa, wv[0], wv[1], wv[2], wv[3]);
                sts_v4(sfb, av[0], av[1], av[2], av[3]);
                if (Cfg::kSfbAtoms > 1 && t.n_mma > 128) {
                    sts_v4(sfb + 512, av[4 % (4 * Cfg::kSfbAtoms)], av[5 % (4 * Cfg::kSfbAtoms)],
                           av[6 % (4 * Cfg::kSfbAtoms)], av[7 % (4 * Cfg::kSfbAtoms)]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar_full_tma + 8 * slot);
            }
        }
        if (Cfg::kScaleWarpsLoadA && !ok) {
            // Gave up (a wait timed out): activation boxes this warp issued
            // may belong to stages nobody consumes, so nothing waits for
            // them; give them time to land before the CTA can exit.
            const uint64_t t0 = ptx::globaltimer_ns();
            while (ptx::globaltimer_ns() - t0 < 50000u) {
            }
        }
    }

    ptx::tc_fence_before();
    if (kCL > 1) {
        __syncwarp();
        ptx::cluster_sync();   // no CTA leaves while others may still write to it
    } else {
        __syncthreads();
    }
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

// The same unit walk as grouped_w4a8_kernel, for a CTA pair: unit = (expert,
// 256 weight rows, token tile).  CTA r of the pair loads weight rows
// [n0 + 128r, +128) and token rows [row0 + r*half, +half); the even CTA's MMA
// thread issues M = 256 MMAs that read both CTAs' shared memory and write
// each CTA's TMEM.  In the odd CTA, the scale warp that owns a ring slot
// tells the even CTA (remote mbarrier arrive) when that stage is loaded; the
// even CTA's commits are multicast to both CTAs' barriers.
template <class Cfg>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Cfg::kThreads, Cfg::kCtasPerSm)
grouped_w4a8_pair_kernel(const __grid_constant__ CUtensorMap map_w,
                         const __grid_constant__ AMaps map_a,
                         const __grid_constant__ CUtensorMap map_out, int out_tma,
                         const uint8_t* __restrict__ a_scale, const uint8_t* __restrict__ w_scale,
                         const int32_t* __restrict__ offsets, int E, int N, int K, int rows,
                         int as_rs, int as_ks, uint16_t* __restrict__ out, uint32_t* status,
                         uint64_t timeout_ns) {
    constexpr int kStages = Cfg::kStages;
    constexpr int kTMax = Cfg::kTMax;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
    const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (sbase - raw_u32);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;

    // Leader (even CTA): bar_full_tma counts both CTAs' TMA bytes of a stage
    // (the odd CTA's loads signal it directly) and takes one arrival from
    // the leader's producer (with the expected bytes) and one from each
    // CTA's scale warp, so the MMA warp waits on one barrier per stage.
    // bar_empty: in both CTAs, released by the leader's multicast commit.
    const uint32_t bar_full_tma = sbase + Cfg::kOffBar;
    const uint32_t bar_empty = bar_full_tma + 8 * kStages;
    const uint32_t bar_tfull = bar_empty + 8 * kStages;
    const uint32_t bar_tempty = bar_tfull + 16;               // leader: both CTAs drained TMEM
    const uint32_t bar_done = bar_tempty + 16;
    // token-scale groups: full (leader, one arrival per CTA), empty (both
    // CTAs, the leader's multicast commit after the group's last MMA)
    const uint32_t bar_sfb_full = bar_done + 8;
    const uint32_t bar_sfb_empty = bar_sfb_full + 8 * Cfg::kSfbSlots;
    volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(base + Cfg::kOffMisc);
    int32_t* s_start = reinterpret_cast<int32_t*>(base + Cfg::kOffSched);
    int32_t* s_rows = s_start + E;
    int32_t* s_ntt = s_rows + E;
    int32_t* s_tile = s_ntt + E;
    int32_t* s_prefix = s_tile + E;   // E + 1 entries

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            ptx::mbar_init(bar_full_tma + 8 * s, 3);
            ptx::mbar_init(bar_empty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_tfull + 8 * b, 1);
            ptx::mbar_init(bar_tempty + 8 * b, 2 * kEpiWarps);
        }
        ptx::mbar_init(bar_done, 1);
        for (int s = 0; s < Cfg::kSfbSlots; ++s) {
            ptx::mbar_init(bar_sfb_full + 8 * s, 2);
            ptx::mbar_init(bar_sfb_empty + 8 * s, 1);
        }
        misc[1] = 0u;   // abort flag
        ptx::fence_barrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(sbase + Cfg::kOffMisc, Cfg::kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&map_w);
        for (int i = 0; i < 4; ++i) ptx::prefetch_tensormap(&map_a.box[i]);
    }

    // Nothing above reads global memory (see grouped_w4a8_kernel).
    ptx::griddep_wait();

    // Per-expert token tiling (tiles rounded to 32 rows: two halves of 16k).
    const int NT = N / (2 * kBW);
    for (int e = threadIdx.x; e < E; e += Cfg::kThreads) {
        const int lo = offsets[e];
        const int hi = offsets[e + 1];
        int r = 0;
        if (lo < 0 || hi < lo || hi > rows) {
            record_error(status, HG_ERR_BAD_OFFSETS, static_cast<uint32_t>(e));
        } else {
            r = hi - lo;
        }
        const int ntt = (r + kTMax - 1) / kTMax;
        const int tile = ntt ? ((((r + ntt - 1) / ntt) + 31) & ~31) : 0;
        s_start[e] = lo;
        s_rows[e] = r;
        s_ntt[e] = ntt;
        s_tile[e] = tile;
        s_prefix[e] = ntt * NT;
    }
    __syncthreads();
    if (warp == 0) {
        // Few rounds: U units dealt to P pairs leave ceil(U/P) * P - U slots
        // of the last round idle.  With at most kPairFillRounds rounds, the
        // experts with the largest tiles (64 rows or more, largest first,
        // then by index) get one token tile more each, NT units per expert,
        // as many as fit in those slots: the round count stays and the
        // largest units shrink (config 3 W2 M = 256: 2.2 rounds, 6 % faster;
        // level to 3 % slower at 8 rounds and more, so not applied there).
        int tiles = 0;
        for (int c = 0; c < E; c += 32) {
            const int e = c + lane;
            tiles += __reduce_add_sync(0xFFFFFFFFu, e < E ? s_ntt[e] : 0);
        }
        const int P = static_cast<int>(gridDim.x >> 1);
        const long long U0 = static_cast<long long>(tiles) * NT;
        const long long rounds = (U0 + P - 1) / P;
        int extra = rounds <= kPairFillRounds ? static_cast<int>((rounds * P - U0) / NT) : 0;
        const uint32_t below = (1u << lane) - 1u;
        uint32_t picked = 0;   // bit c / 32: this lane's expert c + lane got its tile
        for (int v = kTMax; v >= 64 && extra > 0; v -= 32) {
            for (int c = 0; c < E && extra > 0; c += 32) {
                const int e = c + lane;
                bool pick = false;
                int ntt2 = 0, tile2 = 0;
                if (e < E && s_ntt[e] > 0 && s_tile[e] == v && !((picked >> (c >> 5)) & 1u)) {
                    const int r = s_rows[e];
                    ntt2 = s_ntt[e] + 1;
                    tile2 = (((r + ntt2 - 1) / ntt2) + 31) & ~31;
                    pick = tile2 * (ntt2 - 1) < r;   // the last tile keeps a row
                }
                const uint32_t m = __ballot_sync(0xFFFFFFFFu, pick);
                if (pick && __popc(m & below) < extra) {
                    picked |= 1u << (c >> 5);
                    s_ntt[e] = ntt2;
                    s_tile[e] = tile2;
                    s_prefix[e] = ntt2 * NT;
                }
                extra -= min(extra, __popc(m));
            }
        }
        __syncwarp();
        int carry = 0;
        for (int c = 0; c < E; c += 32) {
            const int e = c + lane;
            const int v = e < E ? s_prefix[e] : 0;
            int incl = v;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += y;
            }
            if (e < E) s_prefix[e] = carry + incl - v;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) s_prefix[E] = carry;
    }
    // Barriers and TMEM of both CTAs must exist before either uses the other's.
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    ptx::tc_fence_after();

    const uint32_t tmem_base = misc[0];
    const Sched sch{s_start, s_rows, s_ntt, s_tile, s_prefix, E, NT, 2 * kBW};
    const int U = s_prefix[E];
    constexpr int KB = Cfg::kKB;
    const int KT = K / kBK;   // 128-K blocks
    const int KS = KT / KB;   // stages per unit (K % (128 KB) == 0)
    const WaitCtx wctx{status, misc + 1, timeout_ns};
    // Units u = blockIdx.x / 2 + i * gridDim.x / 2.  The loops read blockIdx
    // and gridDim directly (see the note in grouped_w4a8_kernel on the
    // single-thread roles' sensitivity to values held across them).

    // Unit geometry for this CTA of the pair.
    auto unit_of = [&](int u, int& e, int& wrow0, int& row0, int& nrows, int& n_mma) {
        int lo = 0, hi = E;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (s_prefix[mid] <= u) lo = mid; else hi = mid;
        }
        e = lo;
        const int local = u - s_prefix[lo];
        const int ntt = s_ntt[lo];
        const int nt = local / ntt;
        const int tt = local - nt * ntt;
        const int tile = s_tile[lo];
        wrow0 = nt * 2 * kBW;                      // first weight row of the pair's 256
        row0 = s_start[lo] + tt * tile;
        nrows = min(tile, s_rows[lo] - tt * tile);
        n_mma = (nrows + 31) & ~31;
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer --
        // Whole converged warp; the elected lane issues (see the plain
        // kernel's producer).
        const uint64_t pol_w = ptx::policy_evict_last();   // weight tiles are re-read by the other token tiles of their expert
        const uint32_t full_tma_leader = ptx::mapa_shared(bar_full_tma, 0);
        uint32_t g = 0;
        bool ok = true;
        for (int u = static_cast<int>(blockIdx.x >> 1); ok && u < U;
             u += static_cast<int>(gridDim.x >> 1)) {
            int e, wrow0, row0, nrows, n_mma;
            unit_of(u, e, wrow0, row0, nrows, n_mma);
            const int half = n_mma / 2;
            const int wrow = e * N + wrow0 + static_cast<int>(rank) * kBW;
            for (int ks = 0; ks < KS; ++ks, ++g) {
                const uint32_t slot = g % kStages;
                const uint32_t ph = (g / kStages) & 1u;
                if (!__all_sync(0xFFFFFFFFu, wait_bounded<true>(bar_empty + 8 * slot, ph ^ 1u, wctx,
                                                                kRoleProducer, slot))) {
                    ok = false;
                    break;
                }
                // both CTAs' bytes land on the leader's barrier; the stage's
                // scale warp issues the activation boxes (more warps issuing
                // TMA per SM: measured 1-3 % faster at large M)
                const uint32_t fb = full_tma_leader + 8 * slot;
                if (leader) ptx::mbar_arrive_expect_tx_elect(fb, 2 * KB * (kWTileTx + half * kBK));
#pragma unroll
                for (int j = 0; j < KB; ++j) {
                    ptx::tma_load_2d_pair_elect(
                        sbase + Cfg::kOffW + slot * Cfg::kWStageBytes + j * kWTileBytes, &map_w,
                        (ks * KB + j) * kBK, wrow, fb, pol_w);
                }
            }
        }
        // No copy may land after the CTA exits.  The leader sees its
        // stages complete on bar_full_tma; the odd CTA only through the
        // leader's release of the slot (bar_empty), once it consumed it.
        const uint32_t first = g > kStages ? g - kStages : 0;
        for (uint32_t gg = first; gg < g; ++gg) {
            if (leader) {
                wait_drain(bar_full_tma + 8 * (gg % kStages), (gg / kStages) & 1u, timeout_ns);
            } else {
                // the leader's commit of stage gg completes phase gg / S
                wait_drain(bar_empty + 8 * (gg % kStages), (gg / kStages) & 1u, timeout_ns);
            }
        }
    } else if (warp == 1) {
        if (leader) {
            // --------------------------------------- MMA issuer (pair) ---
            // Whole converged warp of the even CTA; the elected lane issues.
            uint32_t g = 0, tc = 0, gr = 0;   // stages, units, token-scale groups
            bool ok = true;
            for (int u = static_cast<int>(blockIdx.x >> 1); ok && u < U;
                 u += static_cast<int>(gridDim.x >> 1), ++tc) {
                int e, wrow0, row0, nrows, n_mma;
                unit_of(u, e, wrow0, row0, nrows, n_mma);
                const uint32_t b = tc & 1u;
                if (!__all_sync(0xFFFFFFFFu,
                                wait_bounded<true>(bar_tempty + 8 * b, ((tc >> 1) & 1u) ^ 1u, wctx,
                                                   kRoleMma, 0x100u | b))) {
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t idesc0 =
                    ptx::idesc_mxf8f6f4(ptx::kFmtE2M1, ptx::kFmtE4M3, 2 * kBW, n_mma);
                const uint32_t d_tmem = tmem_base + b * Cfg::kAccCols;
                uint32_t gslot = 0, sfb_col = 0;
                for (int ks = 0; ks < KS; ++ks, ++g) {
                    const uint32_t slot = g % kStages;
                    const uint32_t ph = (g / kStages) & 1u;
                    const int kb0 = ks * KB;   // first 128-K block of the stage
                    if ((kb0 & (Cfg::kSfbGroup - 1)) == 0) {
                        // a new token-scale group: both CTAs' words to TMEM
                        gslot = gr % Cfg::kSfbSlots;
                        if (!__all_sync(0xFFFFFFFFu,
                                        wait_bounded<true>(bar_sfb_full + 8 * gslot,
                                                           (gr / Cfg::kSfbSlots) & 1u, wctx,
                                                           kRoleMma, 0x20u | gslot))) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        sfb_col = tmem_base + Cfg::kSfbCol0 + gslot * 4 * Cfg::kSfbAtoms;
                        const uint32_t sfb = sbase + Cfg::kOffSfb + gslot * Cfg::kSfbBytes;
                        ptx::tc_cp_32x128b_warpx4_pair_elect(sfb_col, ptx::desc_sf_32x16(sfb));
                        if (Cfg::kSfbAtoms > 1 && n_mma > 128) {
                            ptx::tc_cp_32x128b_warpx4_pair_elect(sfb_col + 4,
                                                                 ptx::desc_sf_32x16(sfb + 512));
                        }
                    }
                    if (!__all_sync(0xFFFFFFFFu, wait_bounded<true>(bar_full_tma + 8 * slot, ph,
                                                                    wctx, kRoleMma, slot))) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    static_assert(kBK / 32 == 4, "four K = 32 MMAs per 128-K block");
#pragma unroll
                    for (int j = 0; j < KB; ++j) {
                        const uint32_t blk = slot * KB + j;   // ring block
                        const uint32_t sf_col = tmem_base + Cfg::kSfCol0 + blk * 4;
                        const uint64_t sfa = ptx::desc_sf_32x16(sbase + Cfg::kOffSfa + blk * kSfaBytes);
                        const uint64_t wd = ptx::desc_kmajor_sw128(sbase + Cfg::kOffW + blk * kWTileBytes);
                        const uint64_t ad =
                            ptx::desc_kmajor_sw128(sbase + Cfg::kOffA + blk * Cfg::kATileBytes);
                        const uint32_t b_id = static_cast<uint32_t>(kb0 + j) & (Cfg::kSfbGroup - 1);
                        const uint32_t acc = (kb0 + j) != 0 ? 1u : 0u;
                        if (j + 1 < KB) {
                            ptx::pair_kblock_elect(d_tmem, sf_col, sfa, wd, ad,
                                                   ptx::idesc_with_sf_ids(idesc0, 0, b_id),
                                                   ptx::idesc_with_sf_ids(idesc0, 1, b_id),
                                                   ptx::idesc_with_sf_ids(idesc0, 2, b_id),
                                                   ptx::idesc_with_sf_ids(idesc0, 3, b_id), sfb_col, acc);
                        } else {
                            ptx::pair_stage_elect(d_tmem, sf_col, sfa, wd, ad,
                                                  ptx::idesc_with_sf_ids(idesc0, 0, b_id),
                                                  ptx::idesc_with_sf_ids(idesc0, 1, b_id),
                                                  ptx::idesc_with_sf_ids(idesc0, 2, b_id),
                                                  ptx::idesc_with_sf_ids(idesc0, 3, b_id), sfb_col, acc,
                                                  bar_empty + 8 * slot, 0x3);
                        }
                    }
                    const int kb_last = kb0 + KB - 1;
                    if ((kb_last & (Cfg::kSfbGroup - 1)) == Cfg::kSfbGroup - 1 || ks == KS - 1) {
                        // the group's last MMA: its buffer and TMEM columns free once done
                        ptx::tc_commit_pair_multicast_elect(bar_sfb_empty + 8 * gslot, 0x3);
                        ++gr;
                    }
                }
                if (!ok) break;
                ptx::tc_commit_pair_multicast_elect(bar_tfull + 8 * b, 0x3);
            }
            // Everything issued must finish before either CTA releases TMEM.
            ptx::tc_commit_pair_multicast_elect(bar_done, 0x1);
            wait_drain(bar_done, 0u, timeout_ns);
        }
    } else if (warp >= 4 && warp < 4 + kEpiWarps) {
        // ---------------------------------------------------- epilogue --
        const int q = warp & 3;
        const uint32_t tempty_leader = ptx::mapa_shared(bar_tempty, 0);
        const uint32_t out_stage = sbase + Cfg::kOffOut + q * 2 * Cfg::kOutChunkBytes;
        uint32_t out_chunk = 0;
        uint32_t tc = 0;
        for (int u = static_cast<int>(blockIdx.x >> 1); u < U;
             u += static_cast<int>(gridDim.x >> 1), ++tc) {
            int e, wrow0, row0, nrows, n_mma;
            unit_of(u, e, wrow0, row0, nrows, n_mma);
            const uint32_t b = tc & 1u;
            if (!wait_bounded<true>(bar_tfull + 8 * b, (tc >> 1) & 1u, wctx, kRoleEpilogue, b)) break;
            ptx::tc_fence_after();
            const int n_warp = wrow0 + static_cast<int>(rank) * kBW + 32 * q;   // warp's first column
            uint16_t* dst = out + static_cast<size_t>(row0) * N + n_warp + lane;
            const uint32_t taddr =
                tmem_base + (static_cast<uint32_t>(32 * q) << 16) + b * Cfg::kAccCols;
            for (int c0 = 0; c0 < nrows; c0 += 16) {
                uint32_t v[16];
                ptx::tmem_ld_32x32b_x16(taddr + c0, v);
                ptx::tmem_ld_wait();
                if (out_tma && c0 + 16 <= nrows) {
                    // 16 whole rows x this warp's 32 columns: staged in shared
                    // memory and written by one TMA store (rows past the
                    // expert's last row never take this path)
                    const uint32_t buf = out_stage + (out_chunk & 1u) * Cfg::kOutChunkBytes;
                    if (lane == 0) ptx::bulk_wait_group_read<1>();   // this buffer's last store has read it
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        ptx::sts_u16(buf + j * 64 + lane * 2,
                                     __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j]))));
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        ptx::tma_store_2d(&map_out, buf, n_warp, row0 + c0);
                        ptx::bulk_commit_group();
                    }
                    ++out_chunk;
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 + j < nrows) {
                            dst[static_cast<size_t>(c0 + j) * N] =
                                __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[j])));
                        }
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_remote(tempty_leader + 8 * b);
        }
        // every staged store has completed before the CTA can exit
        if (lane == 0) ptx::bulk_wait_group_all();
        __syncwarp();
    } else if (warp == Cfg::kSfbWarp) {
        // ------------------------------------- token-scale staging -----
        // One group of kSfbGroup stages of a unit at a time: word c of lane l
        // holds the scales of token 128a + l + 32c (atom a) at the group's
        // stages, byte j for stage 4m + j (bytes past the unit's last stage,
        // and tokens past the tile, hold 1.0).  Each CTA's TMEM needs the
        // scales of the WHOLE token tile; both CTAs arrive on the leader's
        // group barrier.
        const uint32_t sfb_full_leader = ptx::mapa_shared(bar_sfb_full, 0);
        const bool word_loads = as_ks == 1 && (as_rs & 3) == 0 && (KT & 3) == 0 &&
                                (reinterpret_cast<uintptr_t>(a_scale) & 3u) == 0;
        uint32_t gr = 0;
        bool ok = true;
        for (int u = static_cast<int>(blockIdx.x >> 1); ok && u < U;
             u += static_cast<int>(gridDim.x >> 1)) {
            int e, wrow0, row0, nrows, n_mma;
            unit_of(u, e, wrow0, row0, nrows, n_mma);
            for (int k4 = 0; k4 < KT; k4 += Cfg::kSfbGroup, ++gr) {
                const uint32_t gslot = gr % Cfg::kSfbSlots;
                const int nst = min(Cfg::kSfbGroup, KT - k4);
                uint32_t av[4 * Cfg::kSfbAtoms];
#pragma unroll
                for (int i = 0; i < 4 * Cfg::kSfbAtoms; ++i) {
                    const int tok = 128 * (i >> 2) + lane + 32 * (i & 3);
                    const int r = row0 + tok;
                    uint32_t v = 0x7F7F7F7Fu;
                    if (tok < n_mma && r < rows) {
                        const uint8_t* src = a_scale + static_cast<size_t>(r) * as_rs +
                                             static_cast<size_t>(k4) * as_ks;
                        if (word_loads) {
                            v = __ldg(reinterpret_cast<const uint32_t*>(src));   // 4 whole stages
                        } else {
                            v = 0u;
#pragma unroll
                            for (int j = 0; j < Cfg::kSfbGroup; ++j) {
                                const uint32_t byte =
                                    j < nst ? __ldg(src + static_cast<size_t>(j) * as_ks) : 0x7Fu;
                                v |= byte << (8 * j);
                            }
                        }
                    }
                    av[i] = v;
                }
                if (!__all_sync(0xFFFFFFFFu,
                                wait_bounded<true>(bar_sfb_empty + 8 * gslot,
                                                   ((gr / Cfg::kSfbSlots) & 1u) ^ 1u, wctx,
                                                   kRoleScale, 0x40u | gslot))) {
                    ok = false;
                    break;
                }
                const uint32_t sfb = sbase + Cfg::kOffSfb + gslot * Cfg::kSfbBytes + 16 * lane;
                sts_v4(sfb, av[0], av[1], av[2], av[3]);
                if (Cfg::kSfbAtoms > 1 && n_mma > 128) {
                    sts_v4(sfb + 512, av[4 % (4 * Cfg::kSfbAtoms)], av[5 % (4 * Cfg::kSfbAtoms)],
                           av[6 % (4 * Cfg::kSfbAtoms)], av[7 % (4 * Cfg::kSfbAtoms)]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (leader) {
                        ptx::mbar_arrive(bar_sfb_full + 8 * gslot);
                    } else {
                        ptx::mbar_arrive_remote(sfb_full_leader + 8 * gslot);
                    }
                }
            }
        }
    } else {
        // ------------------------------------------- scale staging -----
        // Weight scales of this CTA's 128 rows, one stage per warp in turn
        // (token scales: the token-scale warp above).
        const int sfw = (warp < 4) ? warp - 2 : warp - 8 + 2;
        const int ws_row = K / 32;
        const uint32_t full_tma_leader = ptx::mapa_shared(bar_full_tma, 0);
        const uint64_t pol_a = ptx::policy_evict_last();
        uint32_t g = 0;
        bool ok = true;
        for (int u = static_cast<int>(blockIdx.x >> 1); ok && u < U;
                 u += static_cast<int>(gridDim.x >> 1)) {
            int e, wrow0, row0, nrows, n_mma;
            unit_of(u, e, wrow0, row0, nrows, n_mma);
            const uint8_t* wsrc =
                w_scale + static_cast<size_t>(e * N + wrow0 + static_cast<int>(rank) * kBW + lane) *
                              ws_row;
            for (int ks = 0; ks < KS; ++ks, ++g) {
                if (static_cast<int>(g % Cfg::kSfWarps) != sfw) continue;
                const uint32_t slot = g % kStages;
                const uint32_t ph = (g / kStages) & 1u;
                uint32_t wv[KB][4];
#pragma unroll
                for (int j = 0; j < KB; ++j) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        wv[j][c] = ldg_u32(wsrc + static_cast<size_t>(32 * c) * ws_row + (ks * KB + j) * 4);
                    }
                }
                if (!__all_sync(0xFFFFFFFFu, wait_bounded<true>(bar_empty + 8 * slot, ph ^ 1u, wctx,
                                                                kRoleScale, slot))) {
                    ok = false;
                    break;
                }
                // this CTA's half of the token tile, counted on the leader's
                // full barrier (armed by the leader's producer for both CTAs)
#pragma unroll
                for (int j = 0; j < KB; ++j) {
                    load_a_rows<true, true>(
                        map_a, sbase + Cfg::kOffA + slot * Cfg::kAStageBytes + j * Cfg::kATileBytes,
                        (ks * KB + j) * kBK, row0 + static_cast<int>(rank) * (n_mma / 2), n_mma / 2,
                        full_tma_leader + 8 * slot, pol_a);
                }
#pragma unroll
                for (int j = 0; j < KB; ++j) {
                    sts_v4(sbase + Cfg::kOffSfa + slot * Cfg::kSfaStageBytes + j * kSfaBytes + 16 * lane,
                           wv[j][0], wv[j][1], wv[j][2], wv[j][3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (leader) {
                        ptx::mbar_arrive(bar_full_tma + 8 * slot);
                    } else {
                        ptx::mbar_arrive_remote(full_tma_leader + 8 * slot);
                    }
                }
            }
        }
        if (!ok) {
            // Gave up (a wait timed out): activation boxes this warp issued
            // may belong to stages nobody consumes, so nothing waits for
            // them; give them time to land before the CTA can exit.
            const uint64_t t0 = ptx::globaltimer_ns();
            while (ptx::globaltimer_ns() - t0 < 50000u) {
            }
        }
    }

    // Neither CTA may release TMEM or shared memory while the pair's MMAs or
    // the other CTA's remote arrivals can still touch them.
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    }
}

__global__ void selftest_wait_kernel(uint32_t* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    const uint32_t b = ptx::smem_u32(&bar);
    if (threadIdx.x == 0) {
        ptx::mbar_init(b, 1);
        abort_flag = 0u;
        ptx::fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const WaitCtx ctx{status, &abort_flag, timeout_ns};
        // Nobody arrives on this barrier: the wait must give up and report.
        wait_bounded(b, 0u, ctx, kRoleSelftest, 0u);
    }
    __syncthreads();
}

// Upper bound on the units of a launch: every non-empty expert needs at most
// ceil(rows_e / T) token tiles <= rows_e / T + 1, times its weight tiles.
long long units_upper(const GemmArgs& a, int t_max, int weight_rows_per_unit) {
    const long long nt = a.N / weight_rows_per_unit;
    const long long active = a.E < a.rows ? a.E : a.rows;
    return ((a.rows + t_max - 1) / t_max + active) * nt;
}

// The occupancy calculator counts any kernel that uses tcgen05 as one CTA
// per SM (measured on GB300: a 320-thread kernel with 100 KB of shared memory
// reads 2 blocks per SM, 1 once it allocates TMEM, while 2 CTAs are resident
// in both cases).  Cluster residency is therefore asked about this stand-in,
// which has the GEMM kernel's block size, shared memory and minimum blocks
// per SM; each GEMM CTA allocates 512 / C TMEM columns, so TMEM never limits
// residency below C per SM.
template <int kThreads, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks) occupancy_stand_in() {}

// Largest number of clusters of `cl` CTAs of `fn` that are resident at once
// (clusters are placed whole inside a GPC, so this can be below
// num_sms * ctas_per_sm / cl).  Cached per kernel, device and shared-memory
// size; 0 when the query fails.
struct ClusterEntry {
    const void* fn;
    int dev;
    int cl;
    size_t smem;
    int value;
};
ClusterEntry g_cluster_cache[32];
int g_cluster_used = 0;
std::mutex g_cluster_mu;

int resident_clusters(const void* fn, int cl, int threads, size_t smem, bool attr_cluster) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(g_cluster_mu);
    for (int i = 0; i < g_cluster_used; ++i) {
        const ClusterEntry& c = g_cluster_cache[i];
        if (c.fn == fn && c.dev == dev && c.cl == cl && c.smem == smem) return c.value;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(cl), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cl);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    if (attr_cluster) {
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    if (g_cluster_used < 32) g_cluster_cache[g_cluster_used++] = ClusterEntry{fn, dev, cl, smem, n};
    return n;
}

// A kernel's dynamic shared-memory limit is a per-device setting: applied
// once per (kernel, device, size) and remembered until gemm_reset_caches.
struct AttrEntry {
    const void* fn;
    int dev;
    size_t bytes;
    cudaError_t err;
};
AttrEntry g_attr_cache[64];
int g_attr_used = 0;
std::mutex g_attr_mu;

template <class Kern>
cudaError_t set_smem_attr(Kern* fn, size_t bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const void* key = reinterpret_cast<const void*>(fn);
    std::lock_guard<std::mutex> lock(g_attr_mu);
    for (int i = 0; i < g_attr_used; ++i) {
        const AttrEntry& c = g_attr_cache[i];
        if (c.fn == key && c.dev == dev && c.bytes == bytes) return c.err;
    }
    const cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(bytes));
    if (err != cudaSuccess) cudaGetLastError();
    if (g_attr_used < 64) g_attr_cache[g_attr_used++] = AttrEntry{key, dev, bytes, err};
    return err;
}

// CTAs one launch uses (0: nothing to do).  Persistent grids: C CTAs per SM,
// as whole clusters and no more clusters than can be resident at once (a
// second wave would idle most of the GPU while it runs), and no more CTAs
// than units (split-K clusters: CL CTAs per unit).
template <class Cfg>
long long grid_plain(const GemmArgs& a) {
    long long grid = static_cast<long long>(a.num_sms) * Cfg::kCtasPerSm;
    const long long u = units_upper(a, Cfg::kTMax, kBW);
    return u < grid ? u : grid;
}

template <class Cfg>
long long grid_cluster(const GemmArgs& a) {
    constexpr int CL = Cfg::kCluster;
    auto* stand_in = occupancy_stand_in<Cfg::kThreads, Cfg::kCtasPerSm>;
    const cudaError_t attr = set_smem_attr(grouped_w4a8_kernel<Cfg>, Cfg::smem_bytes(Cfg::kMaxExperts));
    const cudaError_t attr_s = set_smem_attr(stand_in, kSmemPerBlockMax);
    if (attr != cudaSuccess || attr_s != cudaSuccess) return 0;
    long long grid = static_cast<long long>(a.num_sms) * Cfg::kCtasPerSm / CL * CL;
    const int res = resident_clusters(reinterpret_cast<const void*>(stand_in), CL, Cfg::kThreads,
                                      Cfg::smem_bytes(a.E), true);
    if (res > 0 && static_cast<long long>(res) * CL < grid) grid = static_cast<long long>(res) * CL;
    const long long u = units_upper(a, Cfg::kTMax, kBW) * CL;
    return u < grid ? u : grid;
}

template <class Cfg>
long long grid_pair(const GemmArgs& a) {
    auto* stand_in = occupancy_stand_in<Cfg::kThreads, Cfg::kCtasPerSm>;
    const cudaError_t attr = set_smem_attr(grouped_w4a8_pair_kernel<Cfg>, Cfg::smem_bytes(kMaxE));
    const cudaError_t attr_s = set_smem_attr(stand_in, kSmemPerBlockMax);
    if (attr != cudaSuccess || attr_s != cudaSuccess) return 0;
    long long pairs = static_cast<long long>(a.num_sms / 2) * Cfg::kCtasPerSm;
    const int res = resident_clusters(reinterpret_cast<const void*>(stand_in), 2, Cfg::kThreads,
                                      Cfg::smem_bytes(a.E), true);
    if (res > 0 && res < pairs) pairs = res;
    const long long u = units_upper(a, Cfg::kTMax, 2 * kBW);
    return 2 * (u < pairs ? u : pairs);
}

template <class Cfg>
cudaError_t launch_cfg(const GemmArgs& a, const CUtensorMap& map_w, const AMaps& map_a,
                       cudaStream_t stream) {
    const cudaError_t smem_attr = set_smem_attr(grouped_w4a8_kernel<Cfg>, Cfg::smem_bytes(Cfg::kMaxExperts));
    if (smem_attr != cudaSuccess) return smem_attr;
    const long long grid = grid_plain<Cfg>(a);
    if (grid < 1) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::smem_bytes(a.E);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, grouped_w4a8_kernel<Cfg>, map_w, map_a, a.a_scale, a.w_scale,
                              a.offsets, a.E, a.N, a.K, a.rows, a.as_rs, a.as_ks, a.out, a.status,
                              a.timeout_ns);
}

// Split-K variant: clusters of Cfg::kCluster CTAs, launched with the cluster
// size as a launch attribute.
template <class Cfg>
cudaError_t launch_cluster(const GemmArgs& a, const CUtensorMap& map_w, const AMaps& map_a,
                           cudaStream_t stream) {
    const long long grid = grid_cluster<Cfg>(a);
    if (grid < Cfg::kCluster) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::smem_bytes(a.E);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = Cfg::kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, grouped_w4a8_kernel<Cfg>, map_w, map_a, a.a_scale,
                              a.w_scale, a.offsets, a.E, a.N, a.K, a.rows, a.as_rs, a.as_ks, a.out,
                              a.status, a.timeout_ns);
}

template <class Cfg>
cudaError_t launch_pair(const GemmArgs& a, const CUtensorMap& map_w, const AMaps& map_a,
                        const CUtensorMap* map_out, cudaStream_t stream) {
    const long long grid = grid_pair<Cfg>(a);
    if (grid < 2) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);   // clusters of two: __cluster_dims__
    cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
    cfg.dynamicSmemBytes = Cfg::smem_bytes(a.E);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, grouped_w4a8_pair_kernel<Cfg>, map_w, map_a,
                              map_out ? *map_out : map_w, map_out ? 1 : 0, a.a_scale, a.w_scale,
                              a.offsets, a.E, a.N, a.K, a.rows, a.as_rs, a.as_ks, a.out, a.status,
                              a.timeout_ns);
}

}  // namespace

int gemm_max_experts() { return kMaxE; }

void gemm_reset_caches() {
    {
        std::lock_guard<std::mutex> lock(g_attr_mu);
        g_attr_used = 0;
    }
    std::lock_guard<std::mutex> lock(g_cluster_mu);
    g_cluster_used = 0;
}

int gemm_variant_max_experts(int variant) {
    switch (variant) {
        case 1: return CfgSmall::kMaxExperts;
        case 2: return CfgMid::kMaxExperts;
        case 6: return CfgSplit::kMaxExperts;
        case 8: return CfgWide2::kMaxExperts;
        default: return kMaxE;
    }
}

// Variant choice from the mean rows per expert (the per-expert counts live on
// the device).  Few rows: weight streaming dominates and two small pipelines
// per SM keep the MMA issue rate up; many rows: the widest token tile on CTA
// pairs (256 weight rows x 224 tokens per MMA; measured faster than every
// other shape from ~256 rows per expert up, at every configured size), or,
// when N is not a multiple of 256, 224-row tiles with two CTAs per SM; a
// wave model moves the boundary when the device is known.  With
// at most 32 rows per expert the split-K variant is taken when, counting one
// token tile per active expert (at most min(E, rows) of them), it leaves the
// busiest CTA at least 15 % fewer stages than variant 1 (num_sms = 0: no
// device to ask, never).
int gemm_pick_variant(int32_t E, int32_t N, int32_t K, int32_t rows, int num_sms) {
    const long long per = rows / (E > 0 ? E : 1);
    if (per <= 48) {
        if (num_sms > 0 && rows <= 32LL * E && K >= kBK && N >= kBW) {
            GemmArgs a{};
            a.E = E;
            a.N = N;
            a.K = K;
            a.rows = 1 << 30;      // grid not capped by the unit count
            a.num_sms = num_sms;
            const long long g6 = grid_cluster<CfgSplit>(a);
            const long long g1 = static_cast<long long>(num_sms) * CfgSmall::kCtasPerSm;
            const long long units = static_cast<long long>(E < rows ? E : rows) * (N / kBW);
            const int KT = K / kBK;
            if (g6 >= CfgSplit::kCluster && units > 0) {
                const long long c1 = (units + g1 - 1) / g1 * KT;
                const int s = choose_split(static_cast<int>(units), KT, static_cast<int>(g6),
                                           CfgSplit::kCluster);
                const long long groups = g6 / s;
                const long long c6 = (units + groups - 1) / groups * (KT / s);
                if (20 * c6 <= 17 * c1) return 6;
            }
        }
        return 1;
    }
    // Above 48 rows per expert: variant 2 (112-row tiles, two CTAs per SM)
    // or the large-tile variant (4: CTA pairs; 8 when N % 256 != 0).
    // CTA pairs: a sweep of both variants on every configured shape and on
    // gate/up and down at 80-256 rows per expert (both routings) found the
    // pairs faster from 112 rows per expert up (5-20 %), variant 2 faster or
    // level at 85 rows and below, and a split at 96 (variant 2 9 % faster with
    // balanced experts, the pairs 4 % faster on down): above 100 rows, pairs.
    if (N % (2 * kBW) == 0) return per > 100 ? 4 : 2;
    // Variant 8 (single-CTA 224-row tiles) above 256 rows; at most 256 rows
    // per expert a wave model decides: with every expert at the mean, rounds
    // = units / resident CTAs rounded up, counted in 224-row tiles of 128
    // weight rows over two CTAs per SM; a large-tile round costs 1.25 +
    // 0.0026 * tile rows variant-2 rounds, and the large tile is taken only
    // for a predicted gain of 14 % or more.
    if (per > 256) return 8;
    if (num_sms <= 0 || N < kBW) return 2;
    const long long g = 2LL * num_sms;
    const long long blocks = static_cast<long long>(E) * (N / kBW);
    const long long t2 = (per + CfgMid::kTMax - 1) / CfgMid::kTMax;
    const long long t8 = (per + CfgWide2::kTMax - 1) / CfgWide2::kTMax;
    const long long rows8 = ((per + t8 - 1) / t8 + 15) / 16 * 16;
    const long long c2 = (blocks * t2 + g - 1) / g * 10000;
    const long long c8 = (blocks * t8 + g - 1) / g * (12500 + 26 * rows8);
    return 100 * c8 <= 86 * c2 ? 8 : 2;
}

int gemm_variant_token_tile(int variant) {
    switch (variant) {
        case 1: return CfgSmall::kTMax;
        case 2: return CfgMid::kTMax;
        case 4: return CfgPair::kTMax;
        case 6: return CfgSplit::kTMax;
        case 8: return CfgWide2::kTMax;
        default: return 0;
    }
}

size_t gemm_smem_bytes(int variant, int32_t E) {
    switch (variant) {
        case 1: return CfgSmall::smem_bytes(E);
        case 2: return CfgMid::smem_bytes(E);
        case 4: {   // the larger of the two CTA-pair shapes (which one runs depends on K)
            const size_t a = CfgPair::smem_bytes(E), b = CfgPair2::smem_bytes(E);
            return a > b ? a : b;
        }
        case 6: return CfgSplit::smem_bytes(E);
        default: return CfgWide2::smem_bytes(E);
    }
}

long long gemm_launch_ctas(const GemmArgs& a) {
    switch (a.variant) {
        case 1: return grid_plain<CfgSmall>(a);
        case 2: return grid_plain<CfgMid>(a);
        case 4: return a.K % (CfgPair2::kKB * kBK) == 0 ? grid_pair<CfgPair2>(a) : grid_pair<CfgPair>(a);
        case 6: return grid_cluster<CfgSplit>(a);
        default: return grid_plain<CfgWide2>(a);
    }
}

cudaError_t launch_grouped_gemm(const GemmArgs& a, const CUtensorMap& map_w, const AMaps& map_a,
                                const CUtensorMap* map_out, cudaStream_t stream) {
    switch (a.variant) {
        case 1: return launch_cfg<CfgSmall>(a, map_w, map_a, stream);
        case 2: return launch_cfg<CfgMid>(a, map_w, map_a, stream);
        case 4:   // 256-K stages where K allows (half the MMA warp's waits and commits per MMA)
            return a.K % (CfgPair2::kKB * kBK) == 0
                       ? launch_pair<CfgPair2>(a, map_w, map_a, map_out, stream)
                       : launch_pair<CfgPair>(a, map_w, map_a, map_out, stream);
        case 6: return launch_cluster<CfgSplit>(a, map_w, map_a, stream);
        default: return launch_cfg<CfgWide2>(a, map_w, map_a, stream);
    }
}

cudaError_t launch_selftest_wait(uint32_t* status, uint64_t timeout_ns, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace hg
