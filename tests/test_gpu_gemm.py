"""Grouped W4A8 GEMM on the GPU vs the oracle.

Small cases are compared element by element on the full output; the
configurations' full sizes are compared on whole sampled rows (expert
boundaries, token-tile boundaries, random rows) in the launch configuration
the bench uses.  Tolerance: |gpu - ref| <= 1e-2 |ref| + 1e-2 rms(ref row).
"""
import numpy as np
import pytest
import torch

from oracle import gemm as G
from oracle.plan import plan_expert_offsets
from synth import make_case, make_routing
from synth.inputs import CONFIGS, case_seed, make_acts, make_weights
from tests.gpu_util import assert_rows_close, bf16_bits, np_u8

pytestmark = pytest.mark.gpu

VARIANTS = [1, 2, 4, 6, 8]   # see hg_set_gemm_variant


@pytest.fixture(params=VARIANTS, ids=lambda v: f"variant{v}")
def variant(request, cuda_lib):
    prev = cuda_lib.hg_set_gemm_variant(request.param)
    yield request.param
    cuda_lib.hg_set_gemm_variant(prev)


def _run_gemm(hg, a, a_s, w, w_s, off, out=None):
    dev = "cuda"
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev) if isinstance(x, np.ndarray) else x.to(dev).contiguous()
    o = hg.hg_grouped_w4a8_gemm(t(a), t(a_s), t(w), t(w_s), t(np.asarray(off, dtype=np.int32)),
                                out=out)
    torch.cuda.synchronize()
    return o


def _pack(codes):
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _rand_codes(rng, R, K, E, N, scale_lo=120, scale_hi=134):
    a = rng.integers(0, 256, (R, K), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x3C
    a_s = rng.integers(scale_lo, scale_hi, (R, K // 128), dtype=np.uint8)
    w = rng.integers(0, 256, (E, N, K // 2), dtype=np.uint8)
    w_s = rng.integers(scale_lo, scale_hi, (E, N, K // 32), dtype=np.uint8)
    return a, a_s, w, w_s


def test_config0_full(cuda_lib):
    c = make_case(0, 16)
    ids = torch.from_numpy(c.topk_ids).cuda()
    off_t, _, _ = cuda_lib.hg_plan_expert_offsets(ids, c.E)
    out = cuda_lib.hg_grouped_w4a8_gemm(c.a_fp8.cuda(), c.a_scale.cuda(), c.w_fp4.cuda(),
                                        c.w_scale.cuda(), off_t)
    torch.cuda.synchronize()
    off, *_ = plan_expert_offsets(c.topk_ids, c.E)
    ref = G.grouped_w4a8_gemm(np_u8(c.a_fp8), np_u8(c.a_scale), np_u8(c.w_fp4), np_u8(c.w_scale),
                              off, c.E, c.N, c.K)
    assert_rows_close(bf16_bits(out), ref, "config 0")
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def test_identity_weights(cuda_lib, variant):
    # W = I per expert with unit scales: out = bf16(dequant(A)), exactly
    rng = np.random.default_rng(1)
    E, K = 2, 512
    N = K
    R = 40
    a, a_s, _, _ = _rand_codes(rng, R, K, E, N)
    codes = np.zeros((E, N, K), dtype=np.uint8)
    for e in range(E):
        codes[e, np.arange(N), np.arange(K)] = 0x2
    w = _pack(codes)
    w_s = np.full((E, N, K // 32), 127, dtype=np.uint8)
    off = [0, 17, 40]
    out = _run_gemm(cuda_lib, a, a_s, w, w_s, off)
    ref = G.grouped_w4a8_gemm(a, a_s, w, w_s, off, E, N, K)
    g = bf16_bits(out)
    from oracle.formats import bf16_bits_to_f64
    assert np.array_equal(bf16_bits_to_f64(g), bf16_bits_to_f64(ref))


def test_one_hot_weights_distinct_expert_scales(cuda_lib, variant):
    rng = np.random.default_rng(2)
    E, N, K, R = 3, 256, 1024, 300
    a, a_s, _, _ = _rand_codes(rng, R, K, E, N)
    codes = np.zeros((E, N, K), dtype=np.uint8)
    for e in range(E):
        codes[e, np.arange(N), rng.permutation(K)[:N]] = 0x2
    w = _pack(codes)
    w_s = np.zeros((E, N, K // 32), dtype=np.uint8)
    for e, c in enumerate([-2, 1, 4]):
        w_s[e] = 127 + c
    off = [0, 100, 130, 300]
    out = _run_gemm(cuda_lib, a, a_s, w, w_s, off)
    ref = G.grouped_w4a8_gemm(a, a_s, w, w_s, off, E, N, K)
    from oracle.formats import bf16_bits_to_f64
    assert np.array_equal(bf16_bits_to_f64(bf16_bits(out)), bf16_bits_to_f64(ref))


@pytest.mark.parametrize("E,N,K,cuts", [
    (6, 384, 1024, [0, 1, 17, 17, 240, 470, 700]),        # 1-row, 16-row, empty, 1- and 2-tile experts
    (3, 256, 2048, [0, 224, 225, 673]),                   # exactly one tile, one row, 3 tiles (448 + 1)
    (4, 128, 512, [0, 0, 0, 33, 33]),                     # leading / trailing empty experts
    (2, 512, 3072, [0, 129, 260]),                        # K = 24 stages: the ring wraps many times
    (3, 256, 640, [0, 30, 200, 201]),                     # K = 640: 5 stages (no split divides it)
    (2, 384, 1152, [0, 250, 260]),                        # K = 1152: 9 stages
    (2, 128, 128, [0, 5, 40]),                            # K = 128: a single stage
    (1, 256, 384, [0, 77]),                               # K = 384: 3 stages
    # K % 256 == 0 with 6 and 10 blocks of 128: CTA pairs run 256-K stages whose last
    # token-scale group (four blocks) is half full
    (2, 512, 768, [0, 300, 301]),
    (3, 256, 1280, [0, 60, 290, 291]),
])
def test_ragged_experts_random_codes(cuda_lib, variant, E, N, K, cuts):
    rng = np.random.default_rng(E * 1000 + K)
    R = cuts[-1]
    a, a_s, w, w_s = _rand_codes(rng, R, K, E, N)
    out = _run_gemm(cuda_lib, a, a_s, w, w_s, cuts)
    ref = G.grouped_w4a8_gemm(a, a_s, w, w_s, cuts, E, N, K)
    assert_rows_close(bf16_bits(out), ref, f"ragged E={E} N={N} K={K}")


@pytest.mark.parametrize("N,K", [(128, 512), (256, 512), (256, 384)])
def test_max_experts_mostly_empty(cuda_lib, variant, N, K):
    # 512 experts (the limit), most of them empty, a few with 1..40 rows; with
    # N = 256 the CTA-pair kernels run with their largest schedule tables
    # (256-K stages at K = 512, 128-K stages at K = 384)
    rng = np.random.default_rng(12 + N + K)
    E = 512
    sizes = np.zeros(E, dtype=np.int64)
    hot = rng.choice(E, 24, replace=False)
    sizes[hot] = rng.integers(1, 41, 24)
    cuts = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R = int(cuts[-1])
    a, a_s, w, w_s = _rand_codes(rng, R, K, E, N)
    out = _run_gemm(cuda_lib, a, a_s, w, w_s, cuts)
    ref = G.grouped_w4a8_gemm(a, a_s, w, w_s, cuts, E, N, K)
    assert_rows_close(bf16_bits(out), ref, f"E=512 N={N} K={K}")
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


@pytest.mark.parametrize("E,cuts", [(1, [0, 1]), (2, [0, 0, 1]), (1, [0, 17])])
def test_minimum_shapes(cuda_lib, variant, E, cuts):
    # N = 128 (one weight tile), K = 128 (the smallest supported), one or a few rows
    rng = np.random.default_rng(13 + len(cuts) + cuts[-1])
    N, K = 128, 128
    R = cuts[-1]
    a, a_s, w, w_s = _rand_codes(rng, R, K, E, N)
    out = _run_gemm(cuda_lib, a, a_s, w, w_s, cuts)
    ref = G.grouped_w4a8_gemm(a, a_s, w, w_s, cuts, E, N, K)
    assert_rows_close(bf16_bits(out), ref, f"minimum E={E} rows={R}")


def test_wide_scale_range(cuda_lib, variant):
    rng = np.random.default_rng(5)
    E, N, K, R = 2, 256, 1024, 70
    a, a_s, w, w_s = _rand_codes(rng, R, K, E, N, scale_lo=107, scale_hi=147)
    off = [0, 31, 70]
    out = _run_gemm(cuda_lib, a, a_s, w, w_s, off)
    ref = G.grouped_w4a8_gemm(a, a_s, w, w_s, off, E, N, K)
    assert_rows_close(bf16_bits(out), ref, "wide scales")


def test_guard_rows_untouched(cuda_lib, variant):
    # rows at and beyond off[E] belong to no expert and must not be written
    rng = np.random.default_rng(6)
    E, N, K, R = 3, 256, 512, 100
    a, a_s, w, w_s = _rand_codes(rng, R, K, E, N)
    off = [0, 20, 50, 61]
    out = torch.full((R, N), 12345.0, dtype=torch.bfloat16, device="cuda")
    _run_gemm(cuda_lib, a, a_s, w, w_s, off, out=out)
    canary = torch.tensor(12345.0, dtype=torch.bfloat16).view(torch.int16).item()
    assert np.all(bf16_bits(out[61:]).view(np.int16) == canary)
    ref = G.grouped_w4a8_gemm(a, a_s, w, w_s, off, E, N, K)
    assert_rows_close(bf16_bits(out[:61]), ref[:61], "guard")


def test_deterministic(cuda_lib, variant):
    rng = np.random.default_rng(7)
    E, N, K, R = 4, 512, 2048, 900
    a, a_s, w, w_s = _rand_codes(rng, R, K, E, N)
    off = [0, 100, 400, 401, 900]
    o1 = bf16_bits(_run_gemm(cuda_lib, a, a_s, w, w_s, off))
    o2 = bf16_bits(_run_gemm(cuda_lib, a, a_s, w, w_s, off))
    assert np.array_equal(o1, o2)


def test_bad_offsets_reported(cuda_lib):
    cuda_lib.hg_get_device_status()
    rng = np.random.default_rng(8)
    E, N, K, R = 3, 128, 512, 64
    a, a_s, w, w_s = _rand_codes(rng, R, K, E, N)
    _run_gemm(cuda_lib, a, a_s, w, w_s, [0, 40, 20, 64])     # not monotone
    st, _ = cuda_lib.hg_get_device_status()
    assert st == cuda_lib.HG_ERR_BAD_OFFSETS
    _run_gemm(cuda_lib, a, a_s, w, w_s, [0, 40, 50, 65])     # beyond rows
    st, _ = cuda_lib.hg_get_device_status()
    assert st == cuda_lib.HG_ERR_BAD_OFFSETS
    # the context stays usable
    off = [0, 10, 20, 64]
    out = _run_gemm(cuda_lib, a, a_s, w, w_s, off)
    assert_rows_close(bf16_bits(out), G.grouped_w4a8_gemm(a, a_s, w, w_s, off, E, N, K), "after")
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def test_wait_timeout_is_reported_and_context_survives(cuda_lib):
    cuda_lib.hg_get_device_status()
    cuda_lib.hg_selftest_wait_timeout(20000)        # 20 ms
    st, detail = cuda_lib.hg_get_device_status()
    assert st == cuda_lib.HG_ERR_TIMEOUT
    assert (detail >> 24) == 6
    test_config0_full(cuda_lib)


# --------------------------------------------------------- split-K (variant 6) --

@pytest.mark.parametrize("want", [1, 2, 4])
def test_split_k_each_factor(cuda_lib, want):
    # experts of 1..32 rows (one token tile each) in numbers that make the
    # device pick each split factor for this GPU's resident CTA count
    from fp8_mxfp4_grouped_gb300 import tiles as T
    N, K = 512, 2048
    NT, KT = N // 128, K // 128
    prev = cuda_lib.hg_set_gemm_variant(6)
    try:
        full = cuda_lib.hg_gemm_ctas(512, N, K, 1 << 20)          # grid with units to spare
        assert full > 0 and full % 4 == 0
        E = {1: full, 2: full * 3 // 2, 4: full // 4}[want] // NT
        rng = np.random.default_rng(want)
        cuts = np.concatenate([[0], np.cumsum(rng.integers(1, 33, E))]).astype(np.int32)
        R = int(cuts[-1])
        a, a_s, w, w_s = _rand_codes(rng, R, K, E, N)
        grid = cuda_lib.hg_gemm_ctas(E, N, K, R)
        assert grid == min(full, T.split_grid(10 ** 6, E, N, R))
        assert T.choose_split(E * NT, KT, grid) == want, grid
        o1 = _run_gemm(cuda_lib, a, a_s, w, w_s, cuts)
        o2 = _run_gemm(cuda_lib, a, a_s, w, w_s, cuts)
    finally:
        cuda_lib.hg_set_gemm_variant(prev)
    ref = G.grouped_w4a8_gemm(a, a_s, w, w_s, cuts, E, N, K)
    assert_rows_close(bf16_bits(o1), ref, f"split {want}")
    assert np.array_equal(bf16_bits(o1), bf16_bits(o2))       # fixed summation order
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def test_split_k_auto_choice(cuda_lib):
    # the library's choice on this device equals the host mirror's, and the
    # six-expert-wide W13 projection at one token takes the split variant
    from fp8_mxfp4_grouped_gb300 import tiles as T
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    prev = cuda_lib.hg_set_gemm_variant(6)
    try:
        split_ctas = cuda_lib.hg_gemm_ctas(12, 6144, 3584, 1 << 20)
    finally:
        cuda_lib.hg_set_gemm_variant(prev)
    assert split_ctas > 0
    for E, N, K, rows in [(12, 6144, 3584, 8), (12, 3584, 3072, 8), (12, 6144, 3584, 32),
                          (12, 3584, 3072, 32), (32, 4096, 6144, 512), (4, 256, 512, 32),
                          (12, 6144, 3584, 512), (32, 4096, 6144, 16384),
                          (12, 6144, 3584, 1408), (12, 6144, 3584, 1792), (12, 3584, 3072, 2560),
                          (12, 3584, 3072, 3072), (32, 6144, 2048, 4096), (32, 4096, 6144, 9216),
                          (12, 6144, 3584, 2048)]:
        v = T.pick_variant(E, N, rows, K, sms, split_ctas)
        assert cuda_lib.hg_gemm_token_tile(E, N, K, rows) == T.VARIANT_T_MAX[v], (E, N, K, rows)
    assert T.pick_variant(12, 6144, 8, 3584, sms, split_ctas) == 6


@pytest.mark.parametrize("proj", ["w13", "w2"])
@pytest.mark.parametrize("M", [1, 8])
def test_split_k_config3_small_m(cuda_lib, M, proj):
    prev = cuda_lib.hg_set_gemm_variant(6)
    try:
        test_config3_small_m_full(cuda_lib, M, proj)
    finally:
        cuda_lib.hg_set_gemm_variant(prev)


# ------------------------------------------------ full-size sampled parity --

def _sample_rows(off, rng, t_max, per_expert=3, max_experts=6, pair_n=0):
    """Expert boundaries, token-tile boundaries and random rows of a few experts.
    With pair_n = N (CTA pairs), also the tile boundaries after the pair kernel's
    last-round fill on this device's pairs."""
    from fp8_mxfp4_grouped_gb300.tiles import pair_tiling, token_tiles
    off = np.asarray(off)
    sizes = np.diff(off)
    filled = None
    if pair_n:
        pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
        filled = pair_tiling(sizes, pair_n, pairs)
    nz = np.nonzero(sizes)[0]
    pick = set([int(nz[np.argmax(sizes[nz])]), int(nz[np.argmin(sizes[nz])])])
    pick |= set(int(x) for x in rng.choice(nz, size=min(len(nz), max_experts - 2), replace=False))
    rows = set()
    for e in sorted(pick):
        lo, hi = int(off[e]), int(off[e + 1])
        rows |= {lo, hi - 1}
        # tiles are rounded to 16 rows, or 32 on CTA pairs (224-row tiles)
        for step in ((16, 32) if t_max == 224 else (16,)):
            for r0, valid, _ in token_tiles(hi - lo, t_max, step):
                rows |= {lo + r0, lo + r0 + valid - 1}
        if filled is not None and filled[e][0] > 0:
            n_t, tile = filled[e]
            for tt in range(n_t):
                rows |= {lo + tt * tile, min(hi, lo + (tt + 1) * tile) - 1}
        rows |= set(int(x) for x in rng.integers(lo, hi, per_expert))
    return np.array(sorted(rows), dtype=np.int64)


# Every (configuration, projection, routing, M) of the five workloads except
# the tiny one (whose full output is compared above), grouped so that each
# projection's weights are drawn once.
FULL_CASES = [(cid, M, proj, routing)
              for cid in (1, 2, 3, 4)
              for proj in CONFIGS[cid]["proj"]
              for routing in CONFIGS[cid]["routing"]
              for M in CONFIGS[cid]["Ms"]]


@pytest.mark.parametrize("cid,M,proj,routing", FULL_CASES)
def test_full_size_sampled_rows(cuda_lib, cid, M, proj, routing):
    c = make_case(cid, M, projection=proj, routing=routing, device="cuda")
    ids = torch.from_numpy(c.topk_ids).cuda()
    off_t, _, _ = cuda_lib.hg_plan_expert_offsets(ids, c.E)
    out = cuda_lib.hg_grouped_w4a8_gemm(c.a_fp8, c.a_scale, c.w_fp4, c.w_scale, off_t)
    torch.cuda.synchronize()
    off, *_ = plan_expert_offsets(c.topk_ids, c.E)
    assert np.array_equal(off_t.cpu().numpy(), off)
    rng = np.random.default_rng(cid * 100000 + M)
    t_max = cuda_lib.hg_gemm_token_tile(c.E, c.N, c.K, c.R)
    pair = t_max == 224 and c.N % 256 == 0 and c.R // c.E > 100
    rows = _sample_rows(off, rng, t_max, pair_n=c.N if pair else 0)
    rr = torch.from_numpy(rows).cuda()
    a = c.a_fp8[rr].cpu().numpy()
    a_s = c.a_scale[rr].cpu().numpy()
    # oracle on the sampled rows, re-indexed to a compact problem
    e_of = G.expert_of_rows(off, rows)
    experts = sorted(set(int(x) for x in e_of))
    w = c.w_fp4[experts].cpu().numpy()
    w_s = c.w_scale[experts].cpu().numpy()
    local = np.array([experts.index(int(x)) for x in e_of])
    order = np.argsort(local, kind="stable")
    counts = np.bincount(local, minlength=len(experts))
    loff = np.concatenate([[0], np.cumsum(counts)])
    ref_sorted = G.grouped_w4a8_gemm(a[order], a_s[order], w, w_s, loff, len(experts), c.N, c.K)
    ref = np.empty_like(ref_sorted)
    ref[order] = ref_sorted
    got = bf16_bits(out[rr])
    assert_rows_close(got, ref, f"config {cid} M={M} {c.projection} {c.routing}", row_ids=rows)
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


@pytest.mark.parametrize("proj", ["w13", "w2"])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_config3_small_m_full(cuda_lib, M, proj):
    c = make_case(3, M, projection=proj)
    ids = torch.from_numpy(c.topk_ids).cuda()
    off_t, _, _ = cuda_lib.hg_plan_expert_offsets(ids, c.E)
    out = cuda_lib.hg_grouped_w4a8_gemm(c.a_fp8.cuda(), c.a_scale.cuda(), c.w_fp4.cuda(),
                                        c.w_scale.cuda(), off_t)
    torch.cuda.synchronize()
    off, *_ = plan_expert_offsets(c.topk_ids, c.E)
    ref = G.grouped_w4a8_gemm(np_u8(c.a_fp8), np_u8(c.a_scale), np_u8(c.w_fp4),
                              np_u8(c.w_scale), off, c.E, c.N, c.K)
    assert_rows_close(bf16_bits(out), ref, f"config 3 M={M} {proj}")


def test_graph_capture_replay_matches_eager(cuda_lib):
    c = make_case(0, 16, device="cuda")
    ids = torch.from_numpy(c.topk_ids).cuda()
    E, R = c.E, c.R
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    s2d = torch.empty(R, dtype=torch.int32, device="cuda")
    d2s = torch.empty(R, dtype=torch.int32, device="cuda")
    ws = torch.empty(cuda_lib.hg_plan_workspace_bytes(16, 2, E), dtype=torch.uint8, device="cuda")
    out = torch.empty((R, c.N), dtype=torch.bfloat16, device="cuda")
    def step(stream):
        cuda_lib.hg_plan_expert_offsets(ids, E, off, s2d, d2s, ws, stream=stream)
        cuda_lib.hg_grouped_w4a8_gemm(c.a_fp8, c.a_scale, c.w_fp4, c.w_scale, off, out=out,
                                      stream=stream)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step(s)
    torch.cuda.synchronize()
    eager = bf16_bits(out).copy()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bf16_bits(out), eager)


# ----------------------------------------------------- M-major activation scales --

@pytest.mark.parametrize("E,N,K,cuts", [(6, 384, 1024, [0, 1, 17, 17, 240, 470, 700]),
                                        (2, 512, 3072, [0, 129, 260]),
                                        # 9 stages: CTA pairs stage token scales in groups of
                                        # four, the last group partial
                                        (3, 512, 1152, [0, 100, 100, 333])])
def test_mmajor_scales_ragged(cuda_lib, variant, E, N, K, cuts):
    rng = np.random.default_rng(E * 77 + K)
    R = cuts[-1]
    a, a_s, w, w_s = _rand_codes(rng, R, K, E, N)
    a_mm = np.ascontiguousarray(a_s.T)
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = cuda_lib.hg_grouped_w4a8_gemm_mmajor(t(a), t(a_mm), t(w), t(w_s),
                                               t(np.asarray(cuts, dtype=np.int32)))
    torch.cuda.synchronize()
    ref = G.grouped_w4a8_gemm_mmajor(a, a_mm, w, w_s, cuts, E, N, K)
    assert_rows_close(bf16_bits(out), ref, f"m-major E={E} N={N} K={K}")


@pytest.mark.parametrize("cid,M", [(1, 512), (2, 64), (1, 2048)])
def test_mmajor_matches_row_major_full_size(cuda_lib, cid, M):
    # same codes, scales transposed: the two entry points must agree bit for bit
    # (at M = 2048, CTA pairs: whole-word token-scale loads against byte loads)
    c = make_case(cid, M, device="cuda")
    off, _, _ = cuda_lib.hg_plan_expert_offsets(torch.from_numpy(c.topk_ids).cuda(), c.E)
    o_row = cuda_lib.hg_grouped_w4a8_gemm(c.a_fp8, c.a_scale, c.w_fp4, c.w_scale, off)
    o_mm = cuda_lib.hg_grouped_w4a8_gemm_mmajor(c.a_fp8, c.a_scale.t().contiguous(), c.w_fp4,
                                                c.w_scale, off)
    torch.cuda.synchronize()
    assert torch.equal(o_row.view(torch.int16), o_mm.view(torch.int16))
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def test_shutdown_then_reuse(cuda_lib):
    # after hg_shutdown every per-device setting is queried and applied again
    c = make_case(1, 64)
    ids = torch.from_numpy(c.topk_ids).cuda()
    args = (c.a_fp8.cuda(), c.a_scale.cuda(), c.w_fp4.cuda(), c.w_scale.cuda())
    off, _, _ = cuda_lib.hg_plan_expert_offsets(ids, c.E)
    before = cuda_lib.hg_grouped_w4a8_gemm(*args, off)
    torch.cuda.synchronize()
    cuda_lib.hg_shutdown()
    off2, _, _ = cuda_lib.hg_plan_expert_offsets(ids, c.E)
    after = cuda_lib.hg_grouped_w4a8_gemm(*args, off2)
    torch.cuda.synchronize()
    assert torch.equal(off, off2)
    assert torch.equal(before.view(torch.int16), after.view(torch.int16))
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def _random_problem(seed):
    """A seeded random small problem: expert count, shapes, row counts per
    expert (some empty, some past a tile boundary), codes and scale range."""
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 41))
    N = 128 * int(rng.integers(1, 5))
    K = 128 * int(rng.integers(1, 13))
    sizes = rng.integers(0, 260, E)
    sizes[rng.random(E) < 0.25] = 0
    cuts = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    lo = int(rng.integers(110, 128))
    a, a_s, w, w_s = _rand_codes(rng, int(cuts[-1]), K, E, N, scale_lo=lo, scale_hi=lo + 16)
    return E, N, K, cuts, a, a_s, w, w_s


@pytest.mark.parametrize("seed", range(16))
def test_random_problems_every_variant(cuda_lib, seed):
    # one oracle result per problem, compared with every variant and with the
    # automatic choice
    E, N, K, cuts, a, a_s, w, w_s = _random_problem(9000 + seed)
    ref = G.grouped_w4a8_gemm(a, a_s, w, w_s, cuts, E, N, K)
    prev = cuda_lib.hg_set_gemm_variant(0)
    try:
        for v in [0] + VARIANTS:
            cuda_lib.hg_set_gemm_variant(v)
            out = _run_gemm(cuda_lib, a, a_s, w, w_s, cuts)
            assert_rows_close(bf16_bits(out), ref, f"seed {seed} variant {v} E={E} N={N} K={K}")
    finally:
        cuda_lib.hg_set_gemm_variant(prev)
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def test_tensor_map_cache_same_address_other_shapes(cuda_lib):
    # Encoded tensor maps are cached by (address, shape).  One activation
    # buffer and one weight buffer are reused at the same addresses with other
    # row counts, expert counts and K, and then more distinct buffers than the
    # cache holds are used before the first shape comes back; every call must
    # match the oracle.
    rng = np.random.default_rng(21)
    a_buf = torch.empty(300 * 2048, dtype=torch.uint8, device="cuda")
    w_buf = torch.empty(4 * 256 * 1024, dtype=torch.uint8, device="cuda")

    def run(E, N, K, cuts, seed):
        r = np.random.default_rng(seed)
        R = cuts[-1]
        a, a_s, w, w_s = _rand_codes(r, R, K, E, N)
        av = a_buf[:R * K].view(R, K)
        av.copy_(torch.from_numpy(a))
        wv = w_buf[:E * N * K // 2].view(E, N, K // 2)
        wv.copy_(torch.from_numpy(w))
        out = _run_gemm(cuda_lib, av, a_s, wv, w_s, cuts)
        ref = G.grouped_w4a8_gemm(a, a_s, w, w_s, cuts, E, N, K)
        assert_rows_close(bf16_bits(out), ref, f"cache E={E} N={N} K={K} R={R}")

    shapes = [(3, 256, 1024, [0, 40, 41, 200]), (2, 256, 1024, [0, 150, 300]),
              (4, 128, 2048, [0, 10, 90, 91, 250]), (3, 256, 512, [0, 1, 2, 3])]
    for i, sh in enumerate(shapes):
        run(*sh, seed=100 + i)
        run(*sh, seed=150 + i)      # same address and shape: a cache hit, new contents
    # more distinct activation buffers than the 16 cached entries
    for i in range(20):
        E, N, K, cuts = 1, 128, 512, [0, 16 + i]
        r = np.random.default_rng(200 + i)
        a, a_s, w, w_s = _rand_codes(r, cuts[-1], K, E, N)
        out = _run_gemm(cuda_lib, a, a_s, w, w_s, cuts)
        assert_rows_close(bf16_bits(out), G.grouped_w4a8_gemm(a, a_s, w, w_s, cuts, E, N, K),
                          f"distinct buffer {i}")
    run(*shapes[0], seed=100)
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def test_plan_then_gemm_back_to_back(cuda_lib, variant):
    """Routing plan and GEMM launched back to back on one stream, two routings
    alternating in the same offsets buffer, no host synchronisation: each GEMM
    must read the offsets of the plan just before it (the GEMM is launched with
    programmatic dependent launch, so its set-up runs while that plan is still
    executing).  Each output equals the one from plan, synchronise, GEMM."""
    rng = np.random.default_rng(77)
    E, N, K, M, k = 16, 256, 512, 96, 4
    R = M * k
    a, a_s, w, w_s = _rand_codes(rng, R, K, E, N)
    a_t, as_t, w_t, ws_t = (torch.from_numpy(x).cuda() for x in (a, a_s, w, w_s))
    routings = []
    for skew in (0.0, 3.0):
        p = np.exp(-skew * np.arange(E) / E)
        p /= p.sum()
        ids = np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(M)])
        routings.append(torch.from_numpy(ids.astype(np.int32)).cuda())
    refs = []
    for ids in routings:
        off, _, _ = cuda_lib.hg_plan_expert_offsets(ids, E)
        torch.cuda.synchronize()
        refs.append(cuda_lib.hg_grouped_w4a8_gemm(a_t, as_t, w_t, ws_t, off))
        torch.cuda.synchronize()
    assert not torch.equal(refs[0], refs[1])
    ids_buf = torch.empty_like(routings[0])
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    s2d = torch.empty(R, dtype=torch.int32, device="cuda")
    d2s = torch.empty(R, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(cuda_lib.hg_plan_workspace_bytes(M, k, E), 4), dtype=torch.uint8,
                     device="cuda")
    outs = [torch.empty((R, N), dtype=torch.bfloat16, device="cuda") for _ in range(12)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i, o in enumerate(outs):
            ids_buf.copy_(routings[i % 2])
            cuda_lib.hg_plan_expert_offsets(ids_buf, E, off, s2d, d2s, ws, stream=s)
            cuda_lib.hg_grouped_w4a8_gemm(a_t, as_t, w_t, ws_t, off, out=o, stream=s)
    torch.cuda.synchronize()
    for i, o in enumerate(outs):
        assert torch.equal(o, refs[i % 2]), f"launch {i}"
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK
