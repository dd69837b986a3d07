"""Element formats of the grouped W4A8 GEMM, decoded from their definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

The formats are named by the benchmark command of humming PR #129 ("perf(sm90):
size grouped W4A8 tiles per expert"): activations ``float8e4m3``, weights
``float4e2m1``, block scales ``float8e8m0``, output ``bfloat16``.  The pages
name the formats but do not define them; the definitions below are the
standard ones for those names (OCP microscaling formats and IEEE-style
bfloat16):

* E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit; no inf/NaN.
  Exponent field 0 is subnormal: value m * 2^-1.
* E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 mantissa; no
  infinities; S.1111.111 is NaN; exponent 0 is subnormal: m * 2^-9.
* E8M0: 8-bit unsigned exponent, value 2^(c-127); code 255 is NaN.
* bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa.

All decoding is by 256- or 16-entry float64 tables built once from the
closed forms, so every decoded value is exact.
"""
from __future__ import annotations

import numpy as np


def _e2m1_value(code: int) -> float:
    sign = -1.0 if (code >> 3) & 1 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:
        mag = man * 0.5
    else:
        mag = (1.0 + man / 2.0) * 2.0 ** (exp - 1)
    return sign * mag


def _e4m3_value(code: int) -> float:
    sign = -1.0 if (code >> 7) & 1 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        mag = man * 2.0 ** -9
    else:
        mag = (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return sign * mag


def _e8m0_value(code: int) -> float:
    if code == 255:
        return float("nan")
    return 2.0 ** (code - 127)


#: float64 value of each E2M1 code 0..15 (index = 4-bit code).
E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
#: float64 value of each E4M3 code 0..255.
E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
#: float64 value of each E8M0 code 0..255.
E8M0_TABLE = np.array([_e8m0_value(c) for c in range(256)], dtype=np.float64)


def decode_e2m1_packed(packed: np.ndarray) -> np.ndarray:
    """Decode a packed E2M1 array ``[..., K/2]`` (uint8) to float64 ``[..., K]``.

    Packing reading (the pages do not state it): byte j of a row holds
    element 2j in its low nibble and element 2j+1 in its high nibble.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    lo = packed & 0x0F
    hi = packed >> 4
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.float64)
    out[..., 0::2] = E2M1_TABLE[lo]
    out[..., 1::2] = E2M1_TABLE[hi]
    return out


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    """Decode E4M3 codes (uint8) to float64."""
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def decode_e8m0(codes: np.ndarray) -> np.ndarray:
    """Decode E8M0 scale codes (uint8) to float64 powers of two."""
    return E8M0_TABLE[np.asarray(codes, dtype=np.uint8)]


# --- bfloat16 -------------------------------------------------------------

_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127
_BF16_MIN_NORMAL_EXP = -126
_BF16_MANT_BITS = 7


def round_f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 with round-to-nearest-even, ONCE.

    Going through float32 first would round twice (f64->f32 then f32->bf16)
    and can land on the wrong side of a bf16 tie; this rounds directly from
    float64.  The quantum is 2^(e-7) for a value in binade [2^e, 2^(e+1)),
    floored at 2^-133 below the smallest normal (bf16 subnormals).  Values
    whose rounded magnitude exceeds the largest finite bf16 become +-inf.
    Returns the 16-bit patterns as uint16.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    finite = np.isfinite(x)
    xf = np.where(finite, x, 0.0)
    mag = np.abs(xf)
    _, ex = np.frexp(mag)              # mag = f * 2^ex, f in [0.5, 1)
    e = ex.astype(np.int64) - 1        # mag in [2^e, 2^(e+1))
    e = np.maximum(e, _BF16_MIN_NORMAL_EXP)
    quantum = np.ldexp(1.0, (e - _BF16_MANT_BITS).astype(np.int32))
    q = np.rint(xf / quantum) * quantum            # rint: ties to even
    q = np.where(mag == 0.0, xf, q)                # keep the sign of zero
    overflow = np.abs(q) > _BF16_MAX
    with np.errstate(over="ignore"):
        q32 = q.astype(np.float32)                 # exact: q is a bf16 value
    bits = (q32.view(np.uint32) >> 16).astype(np.uint16)
    bits = np.where(overflow, np.where(q > 0, 0x7F80, 0xFF80), bits).astype(np.uint16)
    # non-finite inputs: keep inf, canonical NaN
    nonfin = ~finite
    if np.any(nonfin):
        xv = x[nonfin]
        nb = np.where(np.isnan(xv), 0x7FC0, np.where(xv > 0, 0x7F80, 0xFF80)).astype(np.uint16)
        bits[nonfin] = nb
    out[...] = bits
    return out


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of bfloat16 bit patterns (uint16)."""
    bits = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    with np.errstate(invalid="ignore"):
        return bits.view(np.float32).astype(np.float64)
