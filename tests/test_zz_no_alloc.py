"""The routing plan that allocates nothing (hg_plan_expert_offsets_noalloc).

Some callers cannot call cudaMalloc at the point where they plan: a host
framework that owns every device allocation through its own memory pool and
does not let a library allocate behind its back, or a latency-critical loop
that cannot take the device-wide synchronisation cudaMalloc and cudaFree may
imply.  For them the plan's workspace is a fixed 256 KiB array inside the
library's device memory.

Only the two-launch plan (more than 32768 routed rows, or count tables too
large for one cluster) touches a workspace, so every shape here takes that
path, which the test asserts through hg_plan_launches.  The shapes are run
back to back, largest first, so each later call finds the array holding an
earlier call's counts; each result must equal both the entry point that takes
a caller-provided workspace and the CPU oracle, bit for bit.  The file is
named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle.plan import plan_expert_offsets

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 256 * 1024


def _bind(lib):
    f = lib.lib.hg_plan_expert_offsets_noalloc
    p = ctypes.c_void_p
    f.argtypes = [p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, p, p, p, p]
    f.restype = ctypes.c_int
    return f


def _noalloc(f, ids, E):
    M, k = ids.shape
    R = M * k
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    s2d = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    d2s = torch.full((R,), -7, dtype=torch.int32, device="cuda")
    st = f(ctypes.c_void_p(ids.data_ptr()), M, k, E, ctypes.c_void_p(off.data_ptr()),
           ctypes.c_void_p(s2d.data_ptr()), ctypes.c_void_p(d2s.data_ptr()),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, off, s2d, d2s


# (M, top_k, E): 157 blocks x 256 experts of counts (160768 bytes, near the
# array's size), then 36 x 200 and 32 x 32 -- all above 32768 routed rows.
SHAPES = [(40000, 8, 256), (9000, 8, 200), (8192, 8, 32), (40000, 8, 256)]


def test_noalloc_plan_matches_workspace_plan_and_oracle(cuda_lib):
    f = _bind(cuda_lib)
    cuda_lib.hg_get_device_status()
    for call, (M, k, E) in enumerate(SHAPES):
        assert cuda_lib.hg_plan_launches(M, k, E) == 2, (M, k, E)
        need = cuda_lib.hg_plan_workspace_bytes(M, k, E)
        assert 0 < need <= SCRATCH_BYTES
        rng = np.random.default_rng(1000 * call + M + E)
        ids_np = rng.integers(0, E, (M, k)).astype(np.int32)
        ids = torch.from_numpy(ids_np).cuda()
        st, off, s2d, d2s = _noalloc(f, ids, E)
        assert st == cuda_lib.HG_OK, (call, st)
        ref = cuda_lib.hg_plan_expert_offsets(ids, E)
        torch.cuda.synchronize()
        for got, want in zip((off, s2d, d2s), ref):
            assert torch.equal(got, want), (call, M, k, E)
        r_off, r_s2d, r_d2s, bad = plan_expert_offsets(ids_np, E)
        assert bad == 0
        assert np.array_equal(off.cpu().numpy(), r_off)
        assert np.array_equal(s2d.cpu().numpy(), r_s2d)
        assert np.array_equal(d2s.cpu().numpy(), r_d2s)
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def test_noalloc_plan_rejects_workspace_beyond_its_array(cuda_lib):
    f = _bind(cuda_lib)
    M, k, E = 40000, 8, 512     # 157 blocks x 512 experts x 4 bytes > 256 KiB
    assert cuda_lib.hg_plan_workspace_bytes(M, k, E) > SCRATCH_BYTES
    ids = torch.zeros((M, k), dtype=torch.int32, device="cuda")
    st, off, _, _ = _noalloc(f, ids, E)
    assert st == cuda_lib.HG_ERR_RESOURCE
    torch.cuda.synchronize()
    assert bool((off == -7).all())          # nothing was launched
