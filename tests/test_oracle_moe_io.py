"""Pins for oracle/moe_io.py (activation quantise + gather, top-k combine)."""
import numpy as np
import torch

from oracle import moe_io as Q
from oracle.formats import decode_e4m3, decode_e8m0, round_f64_to_bf16_bits
from synth import quantize_acts


def _bf16_bits(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_scale_exponent_boundaries():
    # amax exactly 448 * 2^e keeps e; one ulp above moves to e + 1
    for e in (-20, -3, 0, 5, 30):
        a = 448.0 * 2.0 ** e
        assert Q.scale_exponent(a) == e
        assert Q.scale_exponent(np.nextafter(a, np.inf)) == e + 1
        assert Q.scale_exponent(224.0 * 2.0 ** e) == e - 1
        assert Q.scale_exponent(np.nextafter(224.0 * 2.0 ** e, np.inf)) == e
    assert Q.scale_exponent(0.0) == 0
    assert Q.scale_exponent(2.0 ** -140) == -127          # clamped
    assert Q.scale_exponent(1.0) == -8                    # 448 * 2^-9 < 1 <= 448 * 2^-8


def test_e4m3_rne_matches_torch_conversion():
    rng = np.random.default_rng(3)
    q = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 2.0 ** -8,
                        np.array([0.0, -0.0, 448.0, -448.0, 2.0 ** -9, 3 * 2.0 ** -11])])
    q32 = q.astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(q32.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(Q.e4m3_rne(q32), ref)


def test_e4m3_rne_ties_to_even():
    # 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39): even code 0x38
    assert Q.e4m3_rne(np.array([1.0625]))[0] == 0x38
    # 1.1875 halfway between 1.125 (0x39) and 1.25 (0x3A): 0x3A
    assert Q.e4m3_rne(np.array([1.1875]))[0] == 0x3A
    assert Q.e4m3_rne(np.array([-1.1875]))[0] == 0xBA


def test_quantize_rows_closed_forms():
    x = np.zeros((4, 256), dtype=np.float32)
    x[0, :128] = 3.0                     # constant group: scale 2^-7, codes of 384
    x[0, 128:] = 0.0                     # zero group: scale code 127, codes 0
    x[1, :128] = np.linspace(-1, 1, 128)
    x[1, 5] = 448.0                      # amax exactly 448: e = 0
    x[2, 0] = np.inf                     # non-finite group
    x[2, 200] = np.nan
    x[3] = 2.0 ** -120                   # tiny
    codes, scales = Q.quantize_rows(_bf16_bits(x))
    assert scales[0, 0] == 127 - 7 and np.all(decode_e4m3(codes[0, :128]) == 384.0)
    assert scales[0, 1] == 127 and np.all(codes[0, 128:] == 0)
    assert scales[1, 0] == 127 and codes[1, 5] == 0x7E
    assert scales[2, 0] == 0xFF and np.all(codes[2, :128] == 0x7F)
    assert scales[2, 1] == 0xFF and np.all(codes[2, 128:] == 0x7F)
    assert scales[3, 0] == 127 - 127 and np.all(decode_e4m3(codes[3, :128]) * 2.0 ** -127 == 2.0 ** -120)


def test_quantize_rows_agrees_with_the_generator():
    # two independent implementations of the same stated rule
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((32, 512)) * 2.0 ** rng.integers(-12, 12, (32, 1))).astype(np.float32)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    codes, scales = Q.quantize_rows(xb.view(torch.int16).numpy().view(np.uint16))
    g_codes, g_scales = quantize_acts(xb.float())
    assert np.array_equal(scales, g_scales.numpy())
    assert np.array_equal(codes, g_codes.numpy())


def test_quantize_error_bound():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((8, 384)).astype(np.float32)
    xb = _bf16_bits(x)
    codes, scales = Q.quantize_rows(xb)
    xv = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).double().numpy()
    deq = decode_e4m3(codes) * np.repeat(decode_e8m0(scales), 128, axis=1)
    # E4M3 has 3 mantissa bits: relative error <= 2^-4 for normal values
    big = np.abs(xv) >= 2.0 ** -6 * np.repeat(decode_e8m0(scales), 128, axis=1)
    assert np.all(np.abs(deq - xv)[big] <= 2.0 ** -4 * np.abs(xv)[big])


def test_gather_places_tokens():
    x = np.arange(3 * 128, dtype=np.float32).reshape(3, 128) / 64
    s2d = np.array([5, 0, 3, -1, 1, 2], dtype=np.int32)      # top_k = 2: tokens 2,0,1,-,0,1
    a, s = Q.quantize_gather(_bf16_bits(x), 2, s2d)
    codes, scales = Q.quantize_rows(_bf16_bits(x))
    for r, src in enumerate(s2d):
        if src < 0:
            assert np.all(a[r] == 0)
        else:
            assert np.array_equal(a[r], codes[src // 2]) and s[r, 0] == scales[src // 2, 0]


def test_combine_unpermutes_and_weights():
    rng = np.random.default_rng(6)
    M, k, N = 5, 2, 16
    y = rng.standard_normal((M * k, N)).astype(np.float32)
    yb = _bf16_bits(y)
    perm = rng.permutation(M * k).astype(np.int32)
    w = np.tile(np.array([[0.5, 0.25]], dtype=np.float32), (M, 1))
    out = Q.combine_topk(yb, perm, w)
    yv = torch.from_numpy(yb.view(np.int16)).view(torch.bfloat16).double().numpy()
    for t in range(M):
        exact = 0.5 * yv[perm[2 * t]] + 0.25 * yv[perm[2 * t + 1]]      # exact in float64
        assert np.array_equal(out[t], round_f64_to_bf16_bits(exact))
    d = perm.copy()
    d[3] = -1
    out2 = Q.combine_topk(yb, d, w)
    assert np.array_equal(out2[1], round_f64_to_bf16_bits(0.5 * yv[perm[2]]))


def test_scatter_by_hand_and_equal_to_gather_on_a_plan():
    x = np.arange(3 * 128, dtype=np.float32).reshape(3, 128) / 64
    d2s = np.array([4, 1, -1, 0, 5, 9], dtype=np.int32)    # token 1 copy 0 dropped; 9 out of range
    a, s = Q.quantize_scatter(_bf16_bits(x), 2, d2s, np.full((6, 128), 0xAB, np.uint8),
                              np.full((6, 1), 0xCD, np.uint8))
    codes, scales = Q.quantize_rows(_bf16_bits(x))
    want = {4: 0, 1: 0, 0: 1, 5: 2}
    for r in range(6):
        if r in want:
            assert np.array_equal(a[r], codes[want[r]]) and s[r, 0] == scales[want[r], 0]
        else:
            assert np.all(a[r] == 0xAB) and s[r, 0] == 0xCD
    # on a plan's pair of permutations the scatter equals the gather
    from oracle.plan import plan_expert_offsets
    from synth import make_routing
    rng = np.random.default_rng(8)
    M, K, k, E = 40, 256, 4, 6
    xb = _bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
    _, s2d, d2s, _ = plan_expert_offsets(make_routing(M, E, k, "biased", 3), E)
    ga, gs = Q.quantize_gather(xb, k, s2d)
    sa, ss = Q.quantize_scatter(xb, k, d2s)
    assert np.array_equal(ga, sa) and np.array_equal(gs, ss)
