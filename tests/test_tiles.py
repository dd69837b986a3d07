"""Host mirror of the per-expert tile sizer, checked against brute force:
the tiles of an expert cover its rows exactly once, use the fewest tiles any
legal tiling can, and pad at most 15 MMA columns per tile."""
import numpy as np
import pytest

from fp8_mxfp4_grouped_gb300 import tiles as T
from oracle.plan import plan_expert_offsets
from synth import make_routing


@pytest.mark.parametrize("rows", list(range(0, 700)) + [1000, 4096, 14618])
def test_tiles_cover_rows_once(rows):
    ts = T.token_tiles(rows)
    covered = []
    for r0, valid, mma_n in ts:
        assert 0 < valid <= T.T_MAX
        assert mma_n % 16 == 0 and valid <= mma_n <= T.T_MAX and mma_n - valid < 16
        covered.extend(range(r0, r0 + valid))
    assert covered == list(range(rows))
    # fewest tiles: any tiling with tiles of at most T_MAX rows needs ceil(rows / T_MAX)
    assert len(ts) == -(-rows // T.T_MAX)


def test_brute_force_minimal_tile_size():
    # for each row count, the chosen tile is the smallest multiple of 16 that
    # covers the rows with the minimal number of tiles
    for rows in range(1, 1200):
        n_t, tile = T.expert_tiling(rows)
        best = min(t for t in range(16, T.T_MAX + 1, 16) if -(-rows // t) == n_t)
        assert tile == best, rows


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
