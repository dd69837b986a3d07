"""Host mirror of the per-expert tile sizer, checked against brute force:
the tiles of an expert cover its rows exactly once, use the fewest tiles any
legal tiling can, and pad at most 15 MMA columns per tile."""
import numpy as np
import pytest

from fp8_mxfp4_grouped_gb300 import tiles as T
from oracle.plan import plan_expert_offsets
from synth import make_routing


@pytest.mark.parametrize("t_max,step", [(64, 16), (112, 16), (224, 16), (224, 32)])
@pytest.mark.parametrize("rows", list(range(0, 700)) + [1000, 4096, 14618])
def test_tiles_cover_rows_once(rows, t_max, step):
    ts = T.token_tiles(rows, t_max, step)
    covered = []
    for r0, valid, mma_n in ts:
        assert 0 < valid <= t_max
        assert mma_n % step == 0 and valid <= mma_n <= t_max and mma_n - valid < step
        covered.extend(range(r0, r0 + valid))
    assert covered == list(range(rows))
    # fewest tiles: any tiling with tiles of at most t_max rows needs ceil(rows / t_max)
    assert len(ts) == -(-rows // t_max)


@pytest.mark.parametrize("t_max,step", [(64, 16), (112, 16), (224, 16), (224, 32)])
def test_brute_force_minimal_tile_size(t_max, step):
    # for each row count, the chosen tile is the smallest multiple of the MMA
    # step that covers the rows with the minimal number of tiles
    for rows in range(1, 1200):
        n_t, tile = T.expert_tiling(rows, t_max, step)
        best = min(t for t in range(step, t_max + 1, step) if -(-rows // t) == n_t)
        assert tile == best, rows


def test_variant_choice_mirrors_the_library():
    # the choice without a device to ask (no split-K, fixed 256-row
    # boundary); with a device the GPU test of the split-K choice compares
    # the mirror with the device's answers
    import torch
    from fp8_mxfp4_grouped_gb300 import hg
    if torch.cuda.is_available():
        pytest.skip("a device is present: the library's choice depends on it")
    for E in (1, 4, 12, 32, 100, 512):
        for N in (256, 3584, 4096, 6144):
            for rows in (0, 1, 16, 48 * E, 48 * E + E, 256 * E, 256 * E + E, 640 * E, 131072):
                v = T.pick_variant(E, N, rows)
                assert hg.hg_gemm_token_tile(E, N, 6144, rows) == T.VARIANT_T_MAX[v], (E, N, rows)



def test_forced_variant_token_tiles():
    from fp8_mxfp4_grouped_gb300 import hg
    prev = hg.hg_set_gemm_variant(2)
    try:
        assert hg.hg_gemm_token_tile(32, 4096, 6144, 10) == 112
        hg.hg_set_gemm_variant(4)
        assert hg.hg_gemm_token_tile(32, 4096, 6144, 10) == 224
        assert hg.hg_gemm_token_tile(32, 384, 6144, 10) == 224   # falls back to variant 8
        hg.hg_set_gemm_variant(1)
        assert hg.hg_gemm_token_tile(32, 4096, 6144, 10) == 64
        hg.hg_set_gemm_variant(6)
        assert hg.hg_gemm_token_tile(32, 4096, 6144, 10) == 32
        hg.hg_set_gemm_variant(8)
        assert hg.hg_gemm_token_tile(32, 4096, 6144, 10) == 224
    finally:
        hg.hg_set_gemm_variant(prev)
    for removed in (3, 5, 7, 9, -1):
        with pytest.raises(ValueError):
            hg.hg_set_gemm_variant(removed)


@pytest.mark.parametrize("E,N,K,rows,want", [
    (32, 4096, 6144, 2048, 2),    # 64 rows per expert: variant 2 (CTA pairs 9 % slower, measured)
    (32, 4096, 6144, 3072, 2),    # 96 rows: variant 2 (9 % faster with balanced experts)
    (32, 4096, 6144, 3200, 2),    # 100 rows: still variant 2
    (32, 4096, 6144, 3264, 4),    # 102 rows: CTA pairs
    (32, 4096, 6144, 3584, 4),    # 112 rows (gate/up M = 448, measured 5-13 % faster on pairs)
    (32, 4096, 6144, 4096, 4),    # 128 rows (gate/up M = 512)
    (32, 6144, 2048, 6144, 4),    # 192 rows (down M = 768, 11 % faster on pairs)
    (12, 6144, 3584, 2048, 4),    # 170 rows (config 3 W13 M = 256)
    (12, 3584, 3072, 2048, 4),    # 170 rows (config 3 W2 M = 256)
    (12, 3584, 3072, 1024, 2),    # 85 rows (config 3 W2 M = 128, level)
    (32, 4096, 6144, 131072, 4),
    (32, 384, 2048, 131072, 8),   # N % 256 != 0: 224-row tiles on single CTAs above 256 rows
    (32, 384, 2048, 4096, 2),     # N % 256 != 0, 128 rows: variant 2
])
def test_large_tile_variant_choice(E, N, K, rows, want):
    # with N % 256 == 0 the choice depends on the mean rows per expert only;
    # with a device the same (the wave model only guards variant 8)
    assert T.pick_variant(E, N, rows, K, num_sms=152, split_ctas=296) == want
    assert T.pick_variant(E, N, rows, K) == want


def test_tile_inflation_vs_fixed_128():
    # the problem the per-expert sizing addresses: with fixed 128-row tiles,
    # experts just over 128 or 256 rows need a mostly empty extra tile
    ids = make_routing(512, 32, 8, "biased", seed=1512)
    off, *_ = plan_expert_offsets(ids, 32)
    rows = np.diff(off)
    fixed = int(sum(-(-r // 128) for r in rows))
    ours = int(sum(T.expert_tiling(int(r))[0] for r in rows))
    ideal = int(np.count_nonzero(rows))
    assert ours <= fixed
    assert ours >= ideal


def test_units_enumeration():
    off = [0, 3, 3, 300]
    us = T.units(off, 256)
    assert len(us) == 2 * (1 + 2)
    assert {u[0] for u in us} == {0, 2}


@pytest.mark.parametrize("U,KT,G,want", [
    (304, 16, 304, 1),     # one unit per CTA: nothing to even out
    (456, 16, 304, 2),     # 1.5 units per CTA: halves even out (quarters tie, keep 2)
    (76, 16, 304, 4),      # a quarter unit per CTA
    (384, 28, 304, 2),     # 384 weight tiles of 28 stages (six-expert-wide W13 at M=1)
    (224, 24, 304, 4),     # W2 at M=1: 224 tiles of 24 stages
    (608, 48, 304, 1),     # exactly two per CTA
    (0, 8, 304, 1),
    (76, 5, 304, 1),       # K = 640: no split divides 5 stages
    (76, 6, 304, 2),       # K = 768: a quarter of 6 stages is not whole; halves are
    (76, 1, 304, 1),       # K = 128: one stage
    (76, 12, 304, 4),      # K = 1536
])
def test_split_choice(U, KT, G, want):
    assert T.choose_split(U, KT, G) == want
    assert KT % want == 0
    # brute force over the splits that divide the stages: the chosen one
    # gives the least work on the busiest CTA
    def busiest(s):
        return max(len(range(g, U, G // s)) for g in range(G // s)) * (KT // s) if U else 0
    costs = {s: busiest(s) for s in (1, 2, 4) if KT % s == 0}
    assert costs[want] == min(costs.values())
    assert all(costs[s] > costs[want] for s in costs if s < want)


def _pair_units(tiling, N):
    return sum(n for n, _ in tiling) * (N // 256)


@pytest.mark.parametrize("seed", range(40))
def test_pair_fill_keeps_rounds_and_covers_rows(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 40))
    N = 256 * int(rng.integers(1, 30))
    pairs = int(rng.integers(1, 80))
    rows = rng.integers(0, 900, E) * (rng.random(E) < 0.8)
    base = [T.expert_tiling(int(r), 224, 32) for r in rows]
    filled = T.pair_tiling(rows, N, pairs)
    U0, U1 = _pair_units(base, N), _pair_units(filled, N)
    r0 = -(-U0 // pairs)
    assert -(-U1 // pairs) == r0                     # the round count stays
    if r0 > T.PAIR_FILL_ROUNDS:
        assert filled == base
    for r, (n0, t0), (n, t) in zip(rows, base, filled):
        assert n - n0 in (0, 1)                      # at most one extra tile per expert
        if r == 0:
            assert (n, t) == (0, 0)
            continue
        assert t % 32 == 0 and t <= 224 and n * t >= r and (n - 1) * t < r
        if n > n0:
            assert t0 >= 64
    extra = sum(n - n0 for (n0, _), (n, _) in zip(base, filled))
    assert extra * (N // 256) <= r0 * pairs - U0 if r0 <= T.PAIR_FILL_ROUNDS else extra == 0


def test_pair_fill_worked_example():
    # config 3 W2 shape: 12 experts of 170 rows, N = 3584 (14 weight-tile pairs),
    # 76 pairs: 168 units, 3 rounds, 60 idle slots -> 4 experts get a second tile
    got = T.pair_tiling([170] * 12, 3584, 76)
    assert got == [(2, 96)] * 4 + [(1, 192)] * 8
    # largest tiles first, then index; tiles under 64 rows never split
    got = T.pair_tiling([40, 300, 230, 100, 229], 256, 12)
    # base: (1,64) (2,160) (2,128) (1,128) (2,128): 8 units, 1 round, 4 idle -> the
    # 160-row expert, then the three 128-row ones; the 64-row expert stays whole
    assert got == [(1, 64), (3, 128), (3, 96), (2, 64), (3, 96)]
    got = T.pair_tiling([40, 300, 230, 100, 229], 256, 10)
    # 8 units, 1 round of 10: 2 idle -> the 160-row expert, then expert 2 (128, lowest index)
    assert got == [(1, 64), (3, 128), (3, 96), (1, 128), (2, 128)]
    # eight or more rounds: unchanged
    assert T.pair_tiling([170] * 12, 3584, 20) == [(1, 192)] * 12
