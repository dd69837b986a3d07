"""Pins for oracle/plan.py: the hand-derived worked example, planning
invariants, and a loop-by-loop brute force on small inputs."""
import os

import numpy as np
import pytest

from oracle.plan import plan_expert_offsets
from synth import make_routing

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_plan():
    d = {}
    with open(os.path.join(GOLDEN, "plan_example.txt")) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                d[k] = [int(x) for x in v]
    return d


def test_worked_example():
    g = _golden_plan()
    E = g["E"][0]
    ids = np.array(g["topk_ids"], dtype=np.int32).reshape(3, 2)
    off, s2d, d2s, bad = plan_expert_offsets(ids, E)
    assert bad == 0
    assert off.tolist() == g["offsets"]
    assert s2d.tolist() == g["sorted_to_src"]
    assert d2s.tolist() == g["src_to_sorted"]


def check_invariants(ids, E, off, s2d, d2s):
    flat = ids.reshape(-1)
    R = flat.shape[0]
    assert off[0] == 0
    assert np.all(np.diff(off) >= 0)
    assert off[E] == R
    assert sorted(s2d.tolist()) == list(range(R))          # bijection
    assert np.array_equal(d2s[s2d], np.arange(R))          # inverse
    for e in range(E):
        seg = s2d[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e)                      # right expert
        assert np.all(np.diff(seg) > 0)                    # stable


@pytest.mark.parametrize("M,E,k,mode", [(16, 4, 2, "uniform"), (64, 32, 8, "biased"),
                                        (8, 12, 8, "uniform"), (1, 12, 8, "uniform"),
                                        (257, 32, 8, "biased")])
def test_invariants_on_config_shapes(M, E, k, mode):
    ids = make_routing(M, E, k, mode, seed=M + E)
    off, s2d, d2s, bad = plan_expert_offsets(ids, E)
    assert bad == 0
    check_invariants(ids, E, off, s2d, d2s)


def _brute_plan(ids, E):
    flat = [int(x) for x in ids.reshape(-1)]
    counts = [0] * E
    for x in flat:
        counts[x] += 1
    off = [0]
    for c in counts:
        off.append(off[-1] + c)
    s2d, d2s = [], [0] * len(flat)
    for e in range(E):
        for s, x in enumerate(flat):
            if x == e:
                d2s[s] = len(s2d)
                s2d.append(s)
    return off, s2d, d2s


@pytest.mark.parametrize("seed", range(6))
def test_brute_force_with_duplicates(seed):
    # duplicates inside a token are not produced by the generators, but the
    # plan must still be a stable counting sort for them
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 9))
    ids = rng.integers(0, E, (int(rng.integers(1, 12)), int(rng.integers(1, 5)))).astype(np.int32)
    off, s2d, d2s, bad = plan_expert_offsets(ids, E)
    b_off, b_s2d, b_d2s = _brute_plan(ids, E)
    assert bad == 0
    assert off.tolist() == b_off and s2d.tolist() == b_s2d and d2s.tolist() == b_d2s


def test_out_of_range_ids_are_dropped():
    ids = np.array([[0, 5], [-1, 1], [1, 0]], dtype=np.int32)
    off, s2d, d2s, bad = plan_expert_offsets(ids, 2)
    assert bad == 2
    assert off.tolist() == [0, 2, 4]
    assert s2d.tolist() == [0, 5, 3, 4, -1, -1]
    assert d2s.tolist() == [0, -1, -1, 2, 3, 1]


def test_empty_input():
    off, s2d, d2s, bad = plan_expert_offsets(np.zeros((0, 8), dtype=np.int32), 4)
    assert off.tolist() == [0, 0, 0, 0, 0] and s2d.size == 0 and d2s.size == 0 and bad == 0
