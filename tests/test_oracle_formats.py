"""Pins for oracle/formats.py: every code of every format against facts that
do not come from the oracle (literal value lists of the format definitions,
torch's own float8 conversions, hand-derived rounding cases)."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import formats as F

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def test_e2m1_all_codes_match_format_table():
    rows = _read_golden("e2m1_values.txt")
    assert len(rows) == 16
    for code_s, val_s in rows:
        code = int(code_s, 16)
        want = float(val_s)
        got = F.E2M1_TABLE[code]
        assert got == want, (code, got, want)
        assert math.copysign(1.0, got) == math.copysign(1.0, want), code


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.decode_e4m3(np.arange(256, dtype=np.uint8))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_e4m3_landmarks():
    # max normal, min normal, min subnormal (format definition)
    assert F.E4M3_TABLE[0x7E] == 448.0
    assert F.E4M3_TABLE[0x08] == 2.0 ** -6
    assert F.E4M3_TABLE[0x01] == 2.0 ** -9
    assert F.E4M3_TABLE[0x38] == 1.0
    assert F.E4M3_TABLE[0xB8] == -1.0


def test_e8m0_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = F.decode_e8m0(np.arange(256, dtype=np.uint8))
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])
    assert F.E8M0_TABLE[127] == 1.0 and F.E8M0_TABLE[0] == 2.0 ** -127
    assert F.E8M0_TABLE[254] == 2.0 ** 127


def test_e2m1_nibble_order_reading():
    # byte 0x21: low nibble code 1 (0.5) is element 0, high nibble code 2 (1.0) element 1
    got = F.decode_e2m1_packed(np.array([[0x21, 0xF8]], dtype=np.uint8))
    assert got.tolist() == [[0.5, 1.0, -0.0, -6.0]]


def test_bf16_bits_to_f64_matches_torch():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    got = F.bf16_bits_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_round_matches_torch_on_float32_inputs():
    # For float32-representable inputs torch's f32->bf16 conversion rounds once (RNE).
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32) * np.float32(1e3),
        (rng.standard_normal(20000) * 1e-39).astype(np.float32),       # subnormals
        rng.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = F.round_f64_to_bf16_bits(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_round_hand_cases():
    rows = _read_golden("bf16_rounding.txt")
    assert rows
    for x_hex, want_hex in rows:
        x = float.fromhex(x_hex)
        want = int(want_hex, 16)
        got = int(F.round_f64_to_bf16_bits(np.array([x]))[0])
        assert got == want, (x_hex, hex(got), want_hex)


def _bf16_value(b):
    return float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0])


def test_bf16_round_is_nearest_by_brute_force():
    # Independent check: bracket x between consecutive positive bf16 patterns
    # by bisection, then choose the nearer (ties to the even pattern).
    rng = np.random.default_rng(1)
    xs = np.concatenate([rng.standard_normal(300) * 10.0 ** rng.integers(-30, 30, 300),
                         1.0 + rng.integers(0, 2**20, 300) * 2.0 ** -20])
    for x in xs:
        ax = abs(float(x))
        lo, hi = 0, 0x7F7F
        while hi - lo > 1:
            mid = (lo + hi) // 2
            if _bf16_value(mid) <= ax:
                lo = mid
            else:
                hi = mid
        dlo, dhi = ax - _bf16_value(lo), _bf16_value(hi) - ax
        if dlo < dhi or (dlo == dhi and lo % 2 == 0):
            b = lo
        else:
            b = hi
        if x < 0:
            b |= 0x8000
        got = int(F.round_f64_to_bf16_bits(np.array([x]))[0])
        assert got == b, (x, hex(got), hex(b))


def test_bf16_overflow_and_specials():
    r = F.round_f64_to_bf16_bits(np.array([3.4e38, -3.4e38, 3.3e38, np.inf, -np.inf, np.nan, 0.0, -0.0]))
    assert r[0] == 0x7F80 and r[1] == 0xFF80
    assert r[2] == 0x7F78  # 3.3e38 lies between 0x7F78 (3.2964e38) and 0x7F79 (3.3097e38), nearer the first
    assert r[3] == 0x7F80 and r[4] == 0xFF80
    assert (r[5] & 0x7FFF) > 0x7F80
    assert r[6] == 0x0000 and r[7] == 0x8000
