"""The steps on either side of the grouped GEMM: activation quantise + gather,
and the top-k combine.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Quantise (the activation format of humming PR #129's benchmark command --
``float8e4m3`` with ``float8e8m0`` scales per ``--input_scale_group_size
128`` -- produced by a cast like TransformerEngine PR #3459's rowwise MXFP8
cast, description section, with 128-element groups here): per group of 128
values of a row,

    e     = the smallest integer with amax <= 448 * 2^e   (amax = 0 -> e = 0),
            clamped to [-127, 127]
    scale = E8M0 code 127 + e
    codes = E4M3 round-to-nearest-even of x / 2^e

Reading for non-finite inputs (the pages leave them open; the TE review asks
that they be covered): a group holding an Inf or a NaN gets scale code 0xFF
and element codes 0x7F -- the NaN codes of E8M0 and E4M3.

Gather: sorted row r holds token sorted_to_src[r] // top_k (rows with a
negative source stay untouched).  Scatter: token t goes to the rows
src_to_sorted[t*top_k + j] (entries outside [0, M*top_k) skipped).

Combine: out[t, :] = bf16_rne( sum_j w[t, j] * y[src_to_sorted[t*k + j], :] ),
exact sum in float64, terms with src_to_sorted < 0 skipped.
"""
from __future__ import annotations

import numpy as np

from .formats import E4M3_TABLE, bf16_bits_to_f64, round_f64_to_bf16_bits

GROUP = 128
E4M3_MAX = 448.0

# positive finite E4M3 values and their codes, ascending (codes 0x00..0x7E)
_POS_CODES = np.arange(0x00, 0x7F, dtype=np.int64)
_POS_VALUES = E4M3_TABLE[_POS_CODES]


def scale_exponent(amax: float) -> int:
    """Smallest integer e with amax <= 448 * 2^e; 0 for amax == 0; clamped."""
    if amax == 0.0:
        return 0
    e = int(np.floor(np.log2(amax / E4M3_MAX)))
    # settle the inequality exactly (448 * 2^e is exact in float64)
    while amax > E4M3_MAX * 2.0 ** e:
        e += 1
    while e > -1000 and amax <= E4M3_MAX * 2.0 ** (e - 1):
        e -= 1
    return max(-127, min(127, e))


def e4m3_rne(q: np.ndarray) -> np.ndarray:
    """E4M3 codes of values |q| <= 448, round to nearest, ties to the even code."""
    q = np.asarray(q, dtype=np.float64)
    mag = np.abs(q)
    hi = np.searchsorted(_POS_VALUES, mag, side="left")      # first value >= mag
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _POS_VALUES[lo]
    d_hi = _POS_VALUES[hi] - mag
    exact = _POS_VALUES[hi] == mag
    pick_hi = exact | (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo])
    sign = np.where(np.signbit(q), 0x80, 0)     # the sign survives rounding to zero
    return (code | sign).astype(np.uint8)


def quantize_rows(x_bf16_bits: np.ndarray):
    """BF16 bits [M, K] -> (E4M3 codes [M, K], E8M0 codes [M, K/128])."""
    x = bf16_bits_to_f64(np.asarray(x_bf16_bits, dtype=np.uint16))
    M, K = x.shape
    G = K // GROUP
    codes = np.empty((M, K), dtype=np.uint8)
    scales = np.empty((M, G), dtype=np.uint8)
    for m in range(M):
        for g in range(G):
            v = x[m, g * GROUP:(g + 1) * GROUP]
            if not np.all(np.isfinite(v)):
                scales[m, g] = 0xFF
                codes[m, g * GROUP:(g + 1) * GROUP] = 0x7F
                continue
            e = scale_exponent(float(np.max(np.abs(v))))
            scales[m, g] = 127 + e
            codes[m, g * GROUP:(g + 1) * GROUP] = e4m3_rne(v / 2.0 ** e)
    return codes, scales


def quantize_gather(x_bf16_bits, top_k: int, sorted_to_src, a_fp8_init=None, a_scale_init=None):
    """Quantise each token once, then place row r = token sorted_to_src[r] // top_k."""
    codes, scales = quantize_rows(x_bf16_bits)
    s2d = np.asarray(sorted_to_src, dtype=np.int64)
    R = s2d.shape[0]
    K = codes.shape[1]
    a = np.zeros((R, K), dtype=np.uint8) if a_fp8_init is None else np.array(a_fp8_init)
    s = np.zeros((R, K // GROUP), dtype=np.uint8) if a_scale_init is None else np.array(a_scale_init)
    ok = s2d >= 0
    a[ok] = codes[s2d[ok] // top_k]
    s[ok] = scales[s2d[ok] // top_k]
    return a, s


def quantize_scatter(x_bf16_bits, top_k: int, src_to_sorted, a_fp8_init=None, a_scale_init=None):
    """Quantise each token once, then store it to rows src_to_sorted[t*top_k + j]
    (entries outside [0, M*top_k) skipped)."""
    codes, scales = quantize_rows(x_bf16_bits)
    d2s = np.asarray(src_to_sorted, dtype=np.int64)
    M, K = codes.shape
    R = M * top_k
    a = np.zeros((R, K), dtype=np.uint8) if a_fp8_init is None else np.array(a_fp8_init)
    s = np.zeros((R, K // GROUP), dtype=np.uint8) if a_scale_init is None else np.array(a_scale_init)
    for flat in range(R):
        r = int(d2s[flat])
        if 0 <= r < R:
            a[r] = codes[flat // top_k]
            s[r] = scales[flat // top_k]
    return a, s


def combine_topk(y_bf16_bits, src_to_sorted, weights):
    """BF16 bits [M, N] of the weighted sum of each token's expert rows."""
    y = bf16_bits_to_f64(np.asarray(y_bf16_bits, dtype=np.uint16))
    w = np.asarray(weights, dtype=np.float64)
    M, k = w.shape
    d2s = np.asarray(src_to_sorted, dtype=np.int64).reshape(M, k)
    out = np.zeros((M, y.shape[1]), dtype=np.float64)
    for j in range(k):
        ok = d2s[:, j] >= 0
        out[ok] += w[ok, j:j + 1] * y[d2s[ok, j]]
    return round_f64_to_bf16_bits(out)
