"""Helpers shared by the GPU parity tests (not collected as a test module)."""
import numpy as np
import torch

from oracle.formats import bf16_bits_to_f64

# Per-element GEMM tolerance, against the BF16-rounded oracle:
#   |gpu - ref| <= RTOL * |ref| + ROW_RMS_TOL * rms(ref row)
# The GPU accumulates in FP32 and rounds once to BF16; one BF16 ulp is at
# most 2^-8 ~ 0.39% relative, well inside 1%.  A row whose reference is all
# zeros must be exactly zero.
RTOL = 1e-2
ROW_RMS_TOL = 1e-2


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_rows_close(gpu_bits, ref_bits, what="", row_ids=None):
    g = bf16_bits_to_f64(gpu_bits)
    r = bf16_bits_to_f64(ref_bits)
    assert g.shape == r.shape, (g.shape, r.shape)
    rms = np.sqrt(np.mean(r * r, axis=-1, keepdims=True))
    tol = RTOL * np.abs(r) + ROW_RMS_TOL * rms
    err = np.abs(g - r)
    bad = ~(err <= tol)            # also catches NaN on the GPU side
    if bad.any():
        idx = np.argwhere(bad)
        i, j = idx[0]
        rid = row_ids[i] if row_ids is not None else i
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; first at row {rid} "
            f"col {j}: gpu={g[i, j]!r} ref={r[i, j]!r} tol={tol[i, j]!r}; "
            f"rows with errors: {sorted(set(int(row_ids[x] if row_ids is not None else x) for x in idx[:, 0]))[:20]}")


def to_dev(x, device="cuda"):
    if isinstance(x, np.ndarray):
        return torch.from_numpy(np.ascontiguousarray(x)).to(device)
    return x.to(device).contiguous()


def np_u8(t):
    return t.cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
