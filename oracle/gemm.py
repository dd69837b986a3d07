"""Grouped-contiguous FP8 E4M3 x MXFP4 E2M1 GEMM, in float64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

What is computed (humming PR #129, "perf(sm90): size grouped W4A8 tiles per
expert": benchmark command ``--a_dtype float8e4m3 --b_dtype float4e2m1
--c_dtype bfloat16 --bs_dtype float8e8m0 --input_scale_group_size 128
--weight_scale_group_size 32 --gemm_type grouped_contiguous``; first section:
rows routed to one expert are one contiguous range):

    for each expert e and each sorted row r in [off[e], off[e+1]):
        out[r, n] = bf16_rne( sum_k  A(r, k) * W(e, n, k) )
    A(r, k)    = e4m3(a_fp8[r, k])          * 2^(a_scale[r, k // 128] - 127)
    W(e, n, k) = e2m1(w_fp4[e, n, k])       * 2^(w_scale[e, n, k // 32] - 127)

Layouts (readings, the pages give none): a_fp8 [rows, K] row-major;
a_scale [rows, K/128] row-major (the page's default layout; its M-major
variant is a flag); w_fp4 [E, N, K/2] with element 2j in the low nibble of
byte j; w_scale [E, N, K/32]; out [rows, N] bfloat16.  Rows outside every
expert's range (r >= off[E]) are not written by the method; this oracle
leaves them as +0.

Each product of an E4M3 value, an E2M1 value and two powers of two is exact
in float64, and sums of at most a few thousand such terms carry error far
below a bfloat16 ulp, so the result is the exact dot product rounded once.
"""
from __future__ import annotations

import numpy as np

from .formats import (decode_e2m1_packed, decode_e4m3, decode_e8m0,
                      round_f64_to_bf16_bits)

A_GROUP = 128   # --input_scale_group_size
W_GROUP = 32    # --weight_scale_group_size


def dequant_acts(a_fp8: np.ndarray, a_scale: np.ndarray) -> np.ndarray:
    """float64 [rows, K]: E4M3 values times their per-128-K E8M0 scale."""
    vals = decode_e4m3(a_fp8)
    scale = decode_e8m0(a_scale)
    return vals * np.repeat(scale, A_GROUP, axis=-1)


def dequant_weights(w_fp4: np.ndarray, w_scale: np.ndarray) -> np.ndarray:
    """float64 [..., N, K]: E2M1 values times their per-32-K E8M0 scale."""
    vals = decode_e2m1_packed(w_fp4)
    scale = decode_e8m0(w_scale)
    return vals * np.repeat(scale, W_GROUP, axis=-1)


def grouped_w4a8_gemm_f64(a_fp8, a_scale, w_fp4, w_scale, expert_offsets, E, N, K):
    """Unrounded float64 result [rows, N] (rows outside all experts are 0)."""
    a_fp8 = np.asarray(a_fp8, dtype=np.uint8)
    rows = a_fp8.shape[0]
    off = np.asarray(expert_offsets, dtype=np.int64)
    out = np.zeros((rows, N), dtype=np.float64)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi <= lo:
            continue
        a_hat = dequant_acts(a_fp8[lo:hi], np.asarray(a_scale)[lo:hi])
        w_hat = dequant_weights(np.asarray(w_fp4)[e], np.asarray(w_scale)[e])
        out[lo:hi] = a_hat @ w_hat.T
    return out


def grouped_w4a8_gemm(a_fp8, a_scale, w_fp4, w_scale, expert_offsets, E, N, K):
    """BF16 result as uint16 bit patterns [rows, N]."""
    return round_f64_to_bf16_bits(
        grouped_w4a8_gemm_f64(a_fp8, a_scale, w_fp4, w_scale, expert_offsets, E, N, K))


def expert_of_rows(expert_offsets, rows_idx):
    """e(r): the expert whose range holds sorted row r (-1 when none does)."""
    off = np.asarray(expert_offsets, dtype=np.int64)
    r = np.asarray(rows_idx, dtype=np.int64)
    e = np.searchsorted(off, r, side="right") - 1
    E = off.shape[0] - 1
    ok = (e >= 0) & (e < E) & (r < off[-1])
    return np.where(ok, e, -1)


def sampled_outputs(a_fp8, a_scale, w_fp4, w_scale, expert_offsets, rows_idx, cols_idx):
    """BF16 bits of out[r, n] for each pair (rows_idx[i], cols_idx[i]).

    Computes each element on its own: one row of dequantised activations
    times one dequantised weight row of the row's expert.  Pairs whose row
    belongs to no expert give +0.
    """
    r = np.asarray(rows_idx, dtype=np.int64)
    n = np.asarray(cols_idx, dtype=np.int64)
    e = expert_of_rows(expert_offsets, r)
    vals = np.zeros(r.shape[0], dtype=np.float64)
    ok = e >= 0
    if np.any(ok):
        a_hat = dequant_acts(np.asarray(a_fp8)[r[ok]], np.asarray(a_scale)[r[ok]])
        w_hat = dequant_weights(np.asarray(w_fp4)[e[ok], n[ok]],
                                np.asarray(w_scale)[e[ok], n[ok]])
        vals[ok] = np.einsum("ik,ik->i", a_hat, w_hat)
    return round_f64_to_bf16_bits(vals)


def rows_outputs(a_fp8, a_scale, w_fp4, w_scale, expert_offsets, rows_idx):
    """BF16 bits of whole output rows out[r, :] for the sorted rows in rows_idx.

    Groups the requested rows by expert and dequantises each touched
    expert's weights once.  Rows that belong to no expert give +0.
    """
    r = np.asarray(rows_idx, dtype=np.int64)
    e = expert_of_rows(expert_offsets, r)
    N = np.asarray(w_fp4).shape[1]
    vals = np.zeros((r.shape[0], N), dtype=np.float64)
    for ee in np.unique(e[e >= 0]):
        sel = np.nonzero(e == ee)[0]
        a_hat = dequant_acts(np.asarray(a_fp8)[r[sel]], np.asarray(a_scale)[r[sel]])
        w_hat = dequant_weights(np.asarray(w_fp4)[ee], np.asarray(w_scale)[ee])
        vals[sel] = a_hat @ w_hat.T
    return round_f64_to_bf16_bits(vals)


def grouped_w4a8_gemm_mmajor(a_fp8, a_scale_mmajor, w_fp4, w_scale, expert_offsets, E, N, K):
    """BF16 bits of the GEMM with the activation scales stored M-major.

    humming PR #129 benchmark command, option ``--use_m_major_input_scale``:
    the activation scales are laid out ``[K/128, rows]`` (the scale of row r
    for 128-K group g at ``[g, r]``) instead of ``[rows, K/128]``; the method
    is otherwise unchanged.
    """
    a_scale_rows = np.ascontiguousarray(np.asarray(a_scale_mmajor, dtype=np.uint8).T)
    return grouped_w4a8_gemm(a_fp8, a_scale_rows, w_fp4, w_scale, expert_offsets, E, N, K)
