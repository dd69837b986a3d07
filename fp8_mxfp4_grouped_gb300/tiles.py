"""Host mirror of the GEMM kernel's per-expert token tiling.

The kernel builds the same table on the device from expert_offsets (see
``csrc/gemm.cu``); this mirror exists for tests and for the bench's
bookkeeping (units per launch, padded MMA columns).

Rule (humming PR #129, "perf(sm90): size grouped W4A8 tiles per expert",
first section: size the M tile from each expert's own rows so unevenly
routed experts do not pay for mostly empty tiles), restated for the swap-AB
tcgen05 kernel where an expert's tokens are the MMA's N side:

    n_t(e)  = ceil(rows_e / T_MAX)                    token tiles of expert e
    tile(e) = round_up_16(ceil(rows_e / n_t(e)))      rows per token tile
    the last tile of an expert issues MMA N = round_up_16(rows left)

T_MAX depends on the pipeline variant the library picks from rows / E
(``hg_gemm_token_tile``): 64, 112 or 224 (32 for split-K).  With T_MAX = 224 an expert with
130 rows takes one 144-column tile where a fixed 128-row tile would take two.
"""
from __future__ import annotations

T_MAX = 224
VARIANT_T_MAX = {1: 64, 2: 112, 4: 224, 6: 32, 8: 224}
VARIANT_STEP = {1: 16, 2: 16, 4: 32, 6: 16, 8: 16}   # CTA pairs split the token tile in two
SPLIT_CLUSTER = 4        # variant 6: clusters of 4 CTAs, two per SM
MMA_N_STEP = 16
W_TILE = 128


def pick_variant(E: int, N: int, rows: int, K: int = 0, num_sms: int = 0,
                 split_ctas: int = 0) -> int:
    """Mirror of the library's variant choice (mean rows per expert).

    With a device (num_sms > 0, split_ctas = the split-K variant's resident
    CTAs) and at most 32 rows per expert, variant 6 is taken when, counting
    one token tile per active expert, it leaves the busiest CTA at least 15 %
    fewer stages than variant 1.  From 49 rows per expert: with N % 256 == 0,
    CTA pairs (variant 4) above 100 rows per expert and variant 2 below;
    otherwise variant 8 above 256 rows, and from 49 to 256 rows variant 2
    unless a wave model with every expert at the mean predicts a gain of 14 %
    or more for variant 8."""
    per = rows // max(E, 1)
    if per <= 48:
        if num_sms > 0 and rows <= 32 * E and K >= 128 and N >= W_TILE and split_ctas >= SPLIT_CLUSTER:
            units = min(E, rows) * (N // W_TILE)
            KT = K // 128
            if units > 0:
                g1 = num_sms * 2
                c1 = -(-units // g1) * KT
                s = choose_split(units, KT, split_ctas)
                c6 = -(-units // (split_ctas // s)) * (KT // s)
                if 20 * c6 <= 17 * c1:
                    return 6
        return 1
    if N % (2 * W_TILE) == 0:
        return 4 if per > 100 else 2
    if per > 256:
        return 8
    if num_sms <= 0 or N < W_TILE:
        return 2
    # wave model with every expert at the mean, in 224-row tiles of 128
    # weight rows over two CTAs per SM; a variant-8 round costs
    # 1.25 + 0.0026 * tile rows variant-2 rounds; variant 8 only for a
    # predicted gain of 14 % or more
    g = 2 * num_sms
    blocks = E * (N // W_TILE)
    t2 = -(-per // VARIANT_T_MAX[2])
    t8 = -(-per // VARIANT_T_MAX[8])
    rows8 = -(-(-(-per // t8)) // 16) * 16
    c2 = -(-(blocks * t2) // g) * 10000
    c8 = -(-(blocks * t8) // g) * (12500 + 26 * rows8)
    return 8 if 100 * c8 <= 86 * c2 else 2


def expert_tiling(rows_e: int, t_max: int = T_MAX, step: int = MMA_N_STEP):
    """(n_t, tile) for one expert; (0, 0) for an empty expert."""
    if rows_e <= 0:
        return 0, 0
    n_t = -(-rows_e // t_max)
    per = -(-rows_e // n_t)
    tile = -(-per // step) * step
    return n_t, tile


def token_tiles(rows_e: int, t_max: int = T_MAX, step: int = MMA_N_STEP):
    """List of (first_row, valid_rows, mma_n) of one expert's token tiles."""
    n_t, tile = expert_tiling(rows_e, t_max, step)
    out = []
    for tt in range(n_t):
        r0 = tt * tile
        valid = min(tile, rows_e - r0)
        out.append((r0, valid, -(-valid // step) * step))
    return out


PAIR_FILL_ROUNDS = 4     # CTA pairs: last-round fill up to this many rounds


def pair_tiling(rows_per_expert, N: int, pairs: int, t_max: int = T_MAX):
    """Per-expert (n_t, tile) of the CTA-pair kernel (variant 4), with its
    last-round fill: U = sum(n_t) * N/256 units dealt to `pairs` pairs leave
    ceil(U / pairs) * pairs - U slots of the last round idle; with at most
    PAIR_FILL_ROUNDS rounds, floor(idle / (N/256)) experts get one token tile
    more each, taken by tile (64 rows or more, largest first), then by expert
    index, and only where the extra tile leaves the last one a row."""
    step = VARIANT_STEP[4]
    NT = N // (2 * W_TILE)
    til = [list(expert_tiling(int(r), t_max, step)) for r in rows_per_expert]
    U0 = sum(n for n, _ in til) * NT
    rounds = -(-U0 // pairs) if pairs > 0 else 0
    extra = (rounds * pairs - U0) // NT if 0 < rounds <= PAIR_FILL_ROUNDS and NT > 0 else 0
    cands = []
    for e, (n, t) in enumerate(til):
        if n == 0 or t < 64:
            continue
        n2 = n + 1
        t2 = -(-(-(-int(rows_per_expert[e]) // n2)) // step) * step
        if t2 * (n2 - 1) < int(rows_per_expert[e]):
            cands.append((-t, e, n2, t2))
    for _, e, n2, t2 in sorted(cands)[:max(extra, 0)]:
        til[e] = [n2, t2]
    return [tuple(x) for x in til]


def units(offsets, N: int, t_max: int = T_MAX):
    """Work units of one launch: (expert, n0, first sorted row, valid rows, mma_n)."""
    E = len(offsets) - 1
    out = []
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        tiles = token_tiles(hi - lo, t_max)
        for nt in range(N // W_TILE):
            for (r0, valid, mma_n) in tiles:
                out.append((e, nt * W_TILE, lo + r0, valid, mma_n))
    return out


def choose_split(U: int, KT: int, G: int, max_split: int = SPLIT_CLUSTER) -> int:
    """Mirror of the split-K factor variant 6 takes on the device: with G CTAs
    and U units of KT stages, the s in {1, 2, 4} dividing KT that minimises the
    stages of the busiest CTA, ceil(U / (G / s)) * KT / s; ties keep the
    smaller s."""
    best, best_cost = 1, -(-U // G) * KT
    s = 2
    while s <= max_split:
        if KT % s == 0:
            c = -(-U // (G // s)) * (KT // s)
            if c < best_cost:
                best, best_cost = s, c
        s *= 2
    return best


def split_grid(num_sms: int, E: int, N: int, rows: int) -> int:
    """CTAs variant 6 launches: two per SM in whole clusters, capped so that
    every unit can be split four ways."""
    t = VARIANT_T_MAX[6]
    units_max = (-(-rows // t) + min(E, rows)) * (N // W_TILE)
    grid = num_sms * 2 // SPLIT_CLUSTER * SPLIT_CLUSTER
    return min(grid, units_max * SPLIT_CLUSTER)
