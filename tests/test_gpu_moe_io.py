"""The kernels on either side of the GEMM vs the oracle: activation quantise +
gather (bit-exact codes and scales), top-k combine (GEMM tolerance)."""
import numpy as np
import pytest
import torch

from oracle import moe_io as Q
from oracle.plan import plan_expert_offsets
from synth import make_routing
from tests.gpu_util import assert_rows_close, bf16_bits

pytestmark = pytest.mark.gpu


def _tokens(rng, M, K, special=False):
    x = (rng.standard_normal((M, K)) * 2.0 ** rng.integers(-20, 20, (M, 1))).astype(np.float32)
    if special:
        x[0, :128] = 0.0                         # zero group
        x[0, 128:256] = 448.0                    # amax exactly 448 * 2^0
        x[1, 5] = np.inf                         # non-finite groups
        x[1, 300] = -np.inf
        x[2, 130] = np.nan
        x[3, :128] = 2.0 ** -130                 # BF16 subnormals
        x[4, :128] = 3.0e38                      # near the BF16 maximum
        x[5, :] = -1.0 / 3.0
    return torch.from_numpy(x).to(torch.bfloat16)


@pytest.mark.parametrize("M,K,k,E,special", [(3, 128, 2, 4, False), (16, 512, 2, 4, True),
                                             (64, 6144, 8, 32, True), (300, 2048, 8, 32, False)])
def test_quantize_gather_bit_exact(cuda_lib, M, K, k, E, special):
    rng = np.random.default_rng(M * 7 + K)
    x = _tokens(rng, M, K, special)
    ids = make_routing(M, E, k, "biased", M + K)
    _, s2d, _, _ = plan_expert_offsets(ids, E)
    s2d_t = torch.from_numpy(s2d).cuda()
    a, s = cuda_lib.hg_quantize_gather_acts(x.cuda(), k, s2d_t)
    torch.cuda.synchronize()
    ra, rs = Q.quantize_gather(x.view(torch.int16).numpy().view(np.uint16), k, s2d)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(a.cpu().numpy(), ra)


@pytest.mark.parametrize("M,K,k,E,special", [(3, 128, 2, 4, False), (16, 512, 2, 4, True),
                                             (64, 6144, 8, 32, True), (300, 2048, 8, 32, False),
                                             (7, 8192, 1, 3, True)])
def test_quantize_scatter_bit_exact(cuda_lib, M, K, k, E, special):
    rng = np.random.default_rng(M * 11 + K)
    x = _tokens(rng, M, K, special)
    ids = make_routing(M, E, k, "biased", M + 2 * K)
    _, s2d, d2s, _ = plan_expert_offsets(ids, E)
    a, s = cuda_lib.hg_quantize_scatter_acts(x.cuda(), k, torch.from_numpy(d2s).cuda())
    ga, gs = cuda_lib.hg_quantize_gather_acts(x.cuda(), k, torch.from_numpy(s2d).cuda())
    torch.cuda.synchronize()
    ra, rs = Q.quantize_scatter(x.view(torch.int16).numpy().view(np.uint16), k, d2s)
    assert np.array_equal(s.cpu().numpy(), rs) and np.array_equal(a.cpu().numpy(), ra)
    assert torch.equal(a, ga) and torch.equal(s, gs)          # same codes as the gather


def test_quantize_scatter_skips_dropped_and_out_of_range(cuda_lib):
    rng = np.random.default_rng(10)
    M, K, k = 8, 256, 2
    x = _tokens(rng, M, K)
    d2s = np.arange(M * k, dtype=np.int32)[::-1].copy()
    d2s[[3, 9]] = -1
    d2s[12] = M * k + 5                                      # outside the output: skipped
    a = torch.full((M * k, K), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((M * k, K // 128), 0xCD, dtype=torch.uint8, device="cuda")
    cuda_lib.hg_quantize_scatter_acts(x.cuda(), k, torch.from_numpy(d2s).cuda(), a, s)
    torch.cuda.synchronize()
    ra, rs = Q.quantize_scatter(x.view(torch.int16).numpy().view(np.uint16), k, d2s,
                                np.full((M * k, K), 0xAB, np.uint8), np.full((M * k, 2), 0xCD, np.uint8))
    assert np.array_equal(a.cpu().numpy(), ra) and np.array_equal(s.cpu().numpy(), rs)


def test_quantize_gather_skips_dropped_rows(cuda_lib):
    rng = np.random.default_rng(9)
    M, K, k = 8, 256, 2
    x = _tokens(rng, M, K)
    s2d = np.arange(M * k, dtype=np.int32)[::-1].copy()
    s2d[[3, 9, 15]] = -1
    a = torch.full((M * k, K), 0xAB, dtype=torch.uint8, device="cuda")
    s = torch.full((M * k, K // 128), 0xCD, dtype=torch.uint8, device="cuda")
    cuda_lib.hg_quantize_gather_acts(x.cuda(), k, torch.from_numpy(s2d).cuda(), a, s)
    torch.cuda.synchronize()
    ra, rs = Q.quantize_gather(x.view(torch.int16).numpy().view(np.uint16), k, s2d,
                               np.full((M * k, K), 0xAB, np.uint8), np.full((M * k, 2), 0xCD, np.uint8))
    assert np.array_equal(a.cpu().numpy(), ra) and np.array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("M,k,N,E", [(5, 2, 256, 4), (64, 8, 4096, 32), (1000, 8, 6144, 32)])
def test_combine_topk(cuda_lib, M, k, N, E):
    rng = np.random.default_rng(M + N)
    ids = make_routing(M, E, k, "uniform", M)
    _, _, d2s, _ = plan_expert_offsets(ids, E)
    y = torch.from_numpy(rng.standard_normal((M * k, N)).astype(np.float32)).to(torch.bfloat16)
    w = rng.random((M, k)).astype(np.float32)
    w /= w.sum(axis=1, keepdims=True)
    if M > 5:
        d2s = d2s.copy()
        d2s[7] = -1                                          # a dropped id is skipped
    out = cuda_lib.hg_combine_topk(y.cuda(), torch.from_numpy(d2s).cuda(),
                                   torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    ref = Q.combine_topk(y.view(torch.int16).numpy().view(np.uint16), d2s, w)
    assert_rows_close(bf16_bits(out), ref, f"combine M={M} k={k} N={N}")


def test_moe_layer_end_to_end(cuda_lib):
    # tokens -> plan -> quantise+gather -> grouped GEMM -> combine, every step on
    # the GPU, against the oracle chain on the same inputs
    from oracle import gemm as G
    from synth import make_weights
    rng = np.random.default_rng(11)
    M, K, N, E, k = 48, 512, 256, 4, 2
    x = _tokens(rng, M, K)
    ids = make_routing(M, E, k, "uniform", 5)
    w_fp4, w_scale = make_weights(E, N, K, seed=3)
    wts = rng.random((M, k)).astype(np.float32)
    off_t, s2d_t, d2s_t = cuda_lib.hg_plan_expert_offsets(torch.from_numpy(ids).cuda(), E)
    a, s = cuda_lib.hg_quantize_scatter_acts(x.cuda(), k, d2s_t)
    y = cuda_lib.hg_grouped_w4a8_gemm(a, s, w_fp4.cuda(), w_scale.cuda(), off_t)
    out = cuda_lib.hg_combine_topk(y, d2s_t, torch.from_numpy(wts).cuda())
    torch.cuda.synchronize()
    off, s2d, d2s, _ = plan_expert_offsets(ids, E)
    ra, rs = Q.quantize_gather(x.view(torch.int16).numpy().view(np.uint16), k, s2d)
    ry = G.grouped_w4a8_gemm(ra, rs, w_fp4.numpy(), w_scale.numpy(), off, E, N, K)
    ref = Q.combine_topk(ry, d2s, wts)
    assert_rows_close(bf16_bits(out), ref, "MoE layer")


@pytest.mark.parametrize("seed", range(12))
def test_random_problems(cuda_lib, seed):
    # seeded random sizes: both quantisers bit-exact against the oracle (and
    # equal to each other), the combine within the GEMM tolerance
    rng = np.random.default_rng(7000 + seed)
    E = int(rng.integers(1, 65))
    k = int(rng.integers(1, min(E, 8) + 1))
    M = int(rng.integers(1, 401))
    K = 128 * int(rng.integers(1, 17))
    N = 128 * int(rng.integers(1, 33))
    x = _tokens(rng, M, K, special=(seed % 4 == 0 and M >= 6 and K >= 384))
    ids = make_routing(M, E, k, "biased" if seed % 2 else "uniform", 300 + seed)
    _, s2d, d2s, _ = plan_expert_offsets(ids, E)
    xs = x.view(torch.int16).numpy().view(np.uint16)
    a, s = cuda_lib.hg_quantize_scatter_acts(x.cuda(), k, torch.from_numpy(d2s).cuda())
    ga, gs = cuda_lib.hg_quantize_gather_acts(x.cuda(), k, torch.from_numpy(s2d).cuda())
    torch.cuda.synchronize()
    ra, rs = Q.quantize_scatter(xs, k, d2s)
    assert np.array_equal(a.cpu().numpy(), ra) and np.array_equal(s.cpu().numpy(), rs)
    assert torch.equal(a, ga) and torch.equal(s, gs)
    y = torch.from_numpy(rng.standard_normal((M * k, N)).astype(np.float32)).to(torch.bfloat16)
    w = rng.random((M, k)).astype(np.float32)
    out = cuda_lib.hg_combine_topk(y.cuda(), torch.from_numpy(d2s).cuda(),
                                   torch.from_numpy(w).cuda())
    torch.cuda.synchronize()
    ref = Q.combine_topk(y.view(torch.int16).numpy().view(np.uint16), d2s, w)
    assert_rows_close(bf16_bits(out), ref, f"combine seed {seed} M={M} k={k} N={N}")
