"""Pins for oracle/gemm.py against closed forms and an independent brute force.

Each pin is chosen so that a plausible slip in the oracle (a transposed
operand, a wrong group size, a scale applied to the wrong axis, a wrong
expert for a row, a dropped term, double rounding) fails at least one test.
Expected values are computed here with torch's own float8 conversions and
exact Fraction arithmetic, not with the oracle's tables.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import gemm as G
from oracle.formats import bf16_bits_to_f64, round_f64_to_bf16_bits


def _rand_acts(rng, R, K):
    """Random valid E4M3 codes (no NaN) and E8M0 scales near 1."""
    a = rng.integers(0, 256, (R, K), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x3C
    s = rng.integers(127 - 6, 127 + 6, (R, K // 128), dtype=np.uint8)
    return a, s


def _torch_act_values(a, s):
    """float64 dequantised activations from torch's e4m3 / e8m0 conversions."""
    v = torch.from_numpy(a).view(torch.float8_e4m3fn).to(torch.float64)
    sc = torch.from_numpy(s).view(torch.float8_e8m0fnu).to(torch.float64)
    return (v * sc.repeat_interleave(128, dim=1)).numpy()


def _pack(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def _torch_bf16_bits(x64):
    # only used on values exactly representable in float32 (single rounding)
    x32 = x64.astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x64)
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _same_values(x_bits, y_bits):
    """bf16 bit arrays equal as values (+0 == -0: a sum of zeros is +0)."""
    return np.array_equal(bf16_bits_to_f64(x_bits), bf16_bits_to_f64(y_bits))


def test_identity_weights_reproduce_dequantised_activations():
    rng = np.random.default_rng(10)
    E, K = 3, 256
    N = K
    off = np.array([0, 5, 5, 13], dtype=np.int32)    # expert 1 is empty
    R = 13
    a, s = _rand_acts(rng, R, K)
    codes = np.zeros((E, N, K), dtype=np.uint8)
    for e in range(E):
        codes[e, np.arange(N), np.arange(K)] = 0x2          # E2M1 1.0
    w = _pack(codes)
    ws = np.full((E, N, K // 32), 127, dtype=np.uint8)
    got = G.grouped_w4a8_gemm(a, s, w, ws, off, E, N, K)
    want = _torch_bf16_bits(_torch_act_values(a, s))
    assert _same_values(got, want)


def test_one_hot_weights_pin_expert_assignment_and_scales():
    rng = np.random.default_rng(11)
    E, N, K = 4, 128, 512
    off = np.array([0, 3, 9, 9, 20], dtype=np.int32)
    R = 24   # rows 20..23 belong to no expert
    a, s = _rand_acts(rng, R, K)
    codes = np.zeros((E, N, K), dtype=np.uint8)
    perms = [rng.permutation(K)[:N] for _ in range(E)]
    ce = [-3, 0, 2, 5]           # distinct per-expert weight scale exponents
    for e in range(E):
        codes[e, np.arange(N), perms[e]] = 0x2               # 1.0
    w = _pack(codes)
    ws = np.zeros((E, N, K // 32), dtype=np.uint8)
    for e in range(E):
        ws[e] = 127 + ce[e]
    got = G.grouped_w4a8_gemm(a, s, w, ws, off, E, N, K)
    av = _torch_act_values(a, s)
    want = np.zeros((R, N), dtype=np.float64)
    for e in range(E):
        for r in range(off[e], off[e + 1]):
            want[r] = av[r, perms[e]] * 2.0 ** ce[e]
    assert _same_values(got, _torch_bf16_bits(want))


def test_weight_scale_groups_are_32_wide_and_per_column():
    # W = 1.0 everywhere; scale code of group g of column n is 127 + (g + n) % 3.
    rng = np.random.default_rng(12)
    E, N, K = 1, 128, 256
    off = np.array([0, 2], dtype=np.int32)
    a, s = _rand_acts(rng, 2, K)
    w = _pack(np.full((E, N, K), 0x2, dtype=np.uint8))
    ws = np.zeros((E, N, K // 32), dtype=np.uint8)
    for n in range(N):
        for g in range(K // 32):
            ws[0, n, g] = 127 + (g + n) % 3
    got = G.grouped_w4a8_gemm_f64(a, s, w, ws, off, E, N, K)
    av = _torch_act_values(a, s)
    for r in range(2):
        for n in range(N):
            exact = sum(Fraction(float(av[r, k])) * 2 ** ((k // 32 + n) % 3) for k in range(K))
            assert Fraction(float(got[r, n])) == exact


def test_all_ones_weights_give_row_sums():
    rng = np.random.default_rng(13)
    E, N, K = 2, 128, 384
    off = np.array([0, 4, 7], dtype=np.int32)
    a, s = _rand_acts(rng, 7, K)
    w = _pack(np.full((E, N, K), 0x2, dtype=np.uint8))
    ws = np.full((E, N, K // 32), 127, dtype=np.uint8)
    got = G.grouped_w4a8_gemm(a, s, w, ws, off, E, N, K)
    av = _torch_act_values(a, s)
    for r in range(7):
        exact = sum(Fraction(float(v)) for v in av[r])
        want = round_f64_to_bf16_bits(np.array([float(exact)]))[0]
        assert np.all(got[r] == want)


# --- brute force ----------------------------------------------------------

def _bf_e4m3(c):
    s = -1 if c & 0x80 else 1
    e = (c >> 3) & 0xF
    m = c & 7
    if e == 0:
        return s * Fraction(m, 512)
    return s * Fraction(8 + m, 8) * Fraction(2) ** (e - 7)


def _bf_e2m1(c):
    s = -1 if c & 0x8 else 1
    e = (c >> 1) & 3
    m = c & 1
    if e == 0:
        return s * Fraction(m, 2)
    return s * Fraction(2 + m, 2) * Fraction(2) ** (e - 1)


def _bf_bf16_rne(v: Fraction) -> int:
    """Nearest bfloat16 to an exact rational by bisection over bit patterns."""
    def val(b):
        return Fraction(float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0]))
    av = abs(v)
    lo, hi = 0, 0x7F7F
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if val(mid) <= av:
            lo = mid
        else:
            hi = mid
    dlo, dhi = av - val(lo), val(hi) - av
    b = lo if (dlo < dhi or (dlo == dhi and lo % 2 == 0)) else hi
    return b | (0x8000 if v < 0 else 0)


@pytest.mark.parametrize("seed,E,M_rows,K", [(0, 2, 4, 128), (1, 3, 5, 256), (2, 1, 3, 256)])
def test_brute_force_tiny(seed, E, M_rows, K):
    rng = np.random.default_rng(100 + seed)
    N = 128
    a, s = _rand_acts(rng, M_rows, K)
    codes = rng.integers(0, 16, (E, N, K), dtype=np.uint8)
    w = _pack(codes)
    ws = rng.integers(127 - 3, 127 + 3, (E, N, K // 32), dtype=np.uint8)
    cuts = np.sort(rng.integers(0, M_rows + 1, E - 1))
    off = np.concatenate([[0], cuts, [M_rows]]).astype(np.int32)
    got = G.grouped_w4a8_gemm(a, s, w, ws, off, E, N, K)
    for r in range(M_rows):
        e = max(i for i in range(E) if off[i] <= r)
        while off[e + 1] <= r:
            e += 1
        for n in range(0, N, 7):
            acc = Fraction(0)
            for k in range(K):
                byte = int(w[e, n, k // 2])
                nib = (byte & 0xF) if k % 2 == 0 else (byte >> 4)
                aval = _bf_e4m3(int(a[r, k])) * Fraction(2) ** (int(s[r, k // 128]) - 127)
                wval = _bf_e2m1(nib) * Fraction(2) ** (int(ws[e, n, k // 32]) - 127)
                acc += aval * wval
            assert int(got[r, n]) == _bf_bf16_rne(acc), (r, n)


def test_sampled_outputs_equal_full_outputs():
    rng = np.random.default_rng(14)
    E, N, K, R = 3, 256, 256, 20
    a, s = _rand_acts(rng, R, K)
    w = _pack(rng.integers(0, 16, (E, N, K), dtype=np.uint8))
    ws = rng.integers(120, 134, (E, N, K // 32), dtype=np.uint8)
    off = np.array([0, 6, 6, 17], dtype=np.int32)     # rows 17..19 unowned
    full = G.grouped_w4a8_gemm(a, s, w, ws, off, E, N, K)
    rr = rng.integers(0, R, 300)
    cc = rng.integers(0, N, 300)
    samp = G.sampled_outputs(a, s, w, ws, off, rr, cc)
    assert np.array_equal(samp, full[rr, cc])
    assert np.all(full[17:] == 0)


def test_expert_of_rows():
    off = np.array([0, 2, 2, 5], dtype=np.int32)
    assert G.expert_of_rows(off, [0, 1, 2, 3, 4, 5, 9]).tolist() == [0, 0, 2, 2, 2, -1, -1]


def test_rows_outputs_equal_full_outputs():
    rng = np.random.default_rng(15)
    E, N, K, R = 4, 128, 512, 30
    a, s = _rand_acts(rng, R, K)
    w = _pack(rng.integers(0, 16, (E, N, K), dtype=np.uint8))
    ws = rng.integers(120, 134, (E, N, K // 32), dtype=np.uint8)
    off = np.array([0, 9, 9, 20, 27], dtype=np.int32)
    full = G.grouped_w4a8_gemm(a, s, w, ws, off, E, N, K)
    idx = np.array([29, 0, 8, 9, 19, 20, 26, 27, 3])
    assert np.array_equal(G.rows_outputs(a, s, w, ws, off, idx), full[idx])


def test_mmajor_scales_index_groups_by_row():
    # M-major scales: element [g, r]; check against a direct per-element sum
    # written with that indexing (not through the row-major path)
    rng = np.random.default_rng(16)
    E, N, K, R = 2, 128, 256, 6
    a, s_rows = _rand_acts(rng, R, K)
    s_mm = np.ascontiguousarray(s_rows.T)               # [K/128, R]
    w = _pack(rng.integers(0, 16, (E, N, K), dtype=np.uint8))
    ws = rng.integers(124, 131, (E, N, K // 32), dtype=np.uint8)
    off = np.array([0, 4, 6], dtype=np.int32)
    got = G.grouped_w4a8_gemm_mmajor(a, s_mm, w, ws, off, E, N, K)
    for r in range(R):
        e = 0 if r < 4 else 1
        for n in range(0, N, 13):
            acc = Fraction(0)
            for k in range(K):
                byte = int(w[e, n, k // 2])
                nib = (byte & 0xF) if k % 2 == 0 else (byte >> 4)
                acc += (_bf_e4m3(int(a[r, k])) * Fraction(2) ** (int(s_mm[k // 128, r]) - 127)
                        * _bf_e2m1(nib) * Fraction(2) ** (int(ws[e, n, k // 32]) - 127))
            assert int(got[r, n]) == _bf_bf16_rne(acc), (r, n)
