"""Routing plan on the GPU vs the oracle: bit-exact on every configuration's
routing, plus edge cases (empty input, one expert, ids out of range, expert
counts large enough to force a smaller block)."""
import numpy as np
import pytest
import torch

from oracle.plan import plan_expert_offsets
from synth import make_routing
from synth.inputs import CONFIGS, case_seed

pytestmark = pytest.mark.gpu


def _cases():
    out = []
    for cid, cfg in CONFIGS.items():
        for M in cfg["Ms"]:
            for routing in cfg["routing"]:
                out.append((cid, M, routing))
    return out


def _gpu_plan(hg, ids, E):
    t = torch.from_numpy(np.ascontiguousarray(ids)).cuda()
    off, s2d, d2s = hg.hg_plan_expert_offsets(t, E)
    torch.cuda.synchronize()
    return off.cpu().numpy(), s2d.cpu().numpy(), d2s.cpu().numpy()


@pytest.mark.parametrize("cid,M,routing", _cases())
def test_plan_matches_oracle(cuda_lib, cid, M, routing):
    cfg = CONFIGS[cid]
    E, k = cfg["E"], cfg["top_k"]
    ids = make_routing(M, E, k, routing, case_seed(cid, M))
    off, s2d, d2s = _gpu_plan(cuda_lib, ids, E)
    r_off, r_s2d, r_d2s, bad = plan_expert_offsets(ids, E)
    assert bad == 0
    assert np.array_equal(off, r_off)
    assert np.array_equal(s2d, r_s2d)
    assert np.array_equal(d2s, r_d2s)
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


@pytest.mark.parametrize("M,k,E", [(1, 1, 1), (3, 2, 1), (37, 3, 5), (5000, 4, 7), (20000, 8, 64),
                                   (4096, 8, 3000), (2000, 8, 6144)])
def test_plan_random_shapes(cuda_lib, M, k, E):
    rng = np.random.default_rng(M * 7 + E)
    ids = rng.integers(0, E, (M, k)).astype(np.int32)     # duplicates allowed
    off, s2d, d2s = _gpu_plan(cuda_lib, ids, E)
    r_off, r_s2d, r_d2s, _ = plan_expert_offsets(ids, E)
    assert np.array_equal(off, r_off) and np.array_equal(s2d, r_s2d) and np.array_equal(d2s, r_d2s)


def test_plan_empty(cuda_lib):
    t = torch.zeros((0, 8), dtype=torch.int32, device="cuda")
    off, s2d, d2s = cuda_lib.hg_plan_expert_offsets(t, 4)
    assert off.cpu().tolist() == [0] * 5


def test_plan_out_of_range_ids(cuda_lib):
    cuda_lib.hg_get_device_status()
    ids = np.array([[0, 5], [-1, 1], [1, 0]] * 100, dtype=np.int32)
    off, s2d, d2s = _gpu_plan(cuda_lib, ids, 2)
    r_off, r_s2d, r_d2s, bad = plan_expert_offsets(ids, 2)
    assert np.array_equal(off, r_off) and np.array_equal(s2d, r_s2d) and np.array_equal(d2s, r_d2s)
    st, detail = cuda_lib.hg_get_device_status()
    assert st == cuda_lib.HG_ERR_BAD_IDS and detail == bad == 200
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK     # read clears


def test_plan_deterministic(cuda_lib):
    ids = make_routing(16384, 32, 8, "biased", 7)
    a = _gpu_plan(cuda_lib, ids, 32)
    b = _gpu_plan(cuda_lib, ids, 32)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("M,k,E", [
    (512, 8, 32),      # 4096 ids: one CTA
    (4097, 1, 5),      # 4097 ids: two CTAs, the second holding one warp step
    (4096, 8, 33),     # 32768 ids: eight CTAs, four ids per lane
    (32769, 1, 12),    # one id more than one cluster holds: two launches
    (8192, 8, 12),     # 65536 ids: two launches
    (1000, 8, 1500),   # count tables above 48 KB of shared memory
    (3, 3, 2),         # fewer ids than one warp step
])
def test_plan_cluster_boundaries(cuda_lib, M, k, E):
    rng = np.random.default_rng(M + 31 * E)
    ids = rng.integers(0, E, (M, k)).astype(np.int32)
    off, s2d, d2s = _gpu_plan(cuda_lib, ids, E)
    r_off, r_s2d, r_d2s, _ = plan_expert_offsets(ids, E)
    assert np.array_equal(off, r_off) and np.array_equal(s2d, r_s2d) and np.array_equal(d2s, r_d2s)


def test_plan_out_of_range_ids_across_ctas(cuda_lib):
    # dropped ids in every CTA of a multi-CTA plan: rows past off[E] are -1
    cuda_lib.hg_get_device_status()
    rng = np.random.default_rng(5)
    ids = rng.integers(-2, 14, (2500, 8)).astype(np.int32)     # E = 12: -2, -1, 12, 13 dropped
    off, s2d, d2s = _gpu_plan(cuda_lib, ids, 12)
    r_off, r_s2d, r_d2s, bad = plan_expert_offsets(ids, 12)
    assert bad > 0
    assert np.array_equal(off, r_off) and np.array_equal(s2d, r_s2d) and np.array_equal(d2s, r_d2s)
    st, detail = cuda_lib.hg_get_device_status()
    assert st == cuda_lib.HG_ERR_BAD_IDS and detail == bad


def test_plan_launch_count(cuda_lib):
    assert cuda_lib.hg_plan_launches(0, 8, 32) == 0
    assert cuda_lib.hg_plan_launches(64, 8, 32) == 1
    assert cuda_lib.hg_plan_launches(4096, 8, 32) == 1          # 32768 ids: one cluster
    assert cuda_lib.hg_plan_launches(4097, 8, 32) == 2
    assert cuda_lib.hg_plan_launches(1000, 8, 3000) == 2        # count tables beyond one CTA
    assert cuda_lib.hg_plan_launches(-1, 8, 32) == -1


@pytest.mark.parametrize("seed", range(24))
def test_plan_random_problems(cuda_lib, seed):
    # seeded random sizes across the one-cluster and two-launch paths, some
    # ids out of range; bit-exact against the oracle
    rng = np.random.default_rng(5000 + seed)
    E = int(rng.choice([1, 3, 12, 32, 64, 200, 2000]))
    k = int(rng.integers(1, min(E, 8) + 1))
    M = int(rng.choice([1, 7, 100, 513, 4096, 9000, 20000]))
    ids = rng.integers(0, E, (M, k)).astype(np.int32)
    if seed % 3 == 0:
        drop = rng.random((M, k)) < 0.05
        ids[drop] = rng.choice([-1, E, E + 5], int(drop.sum()))
    cuda_lib.hg_get_device_status()
    off, s2d, d2s = _gpu_plan(cuda_lib, ids, E)
    r_off, r_s2d, r_d2s, bad = plan_expert_offsets(ids, E)
    assert np.array_equal(off, r_off) and np.array_equal(s2d, r_s2d) and np.array_equal(d2s, r_d2s)
    st, detail = cuda_lib.hg_get_device_status()
    assert (st, detail) == ((cuda_lib.HG_ERR_BAD_IDS, bad) if bad else (cuda_lib.HG_OK, 0))
