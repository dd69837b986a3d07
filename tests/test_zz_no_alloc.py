"""The allocation-free routing plan (hg_plan_expert_offsets_noalloc).

It exists for callers that cannot call cudaMalloc where they plan (inside a
CUDA-graph capture, under a host that owns all device memory, or in loops
that cannot take cudaMalloc's implicit synchronisation): its workspace is a
fixed 256 KiB array inside the library.  This test calls it through the C ABI
twice in a row, on shapes that take the two-launch path (the one that uses
the workspace), and requires bit-identical results to the entry point that
takes a caller-provided workspace.  It is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


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


@pytest.mark.parametrize("M,k,E", [(4096, 8, 32), (2500, 8, 200)])
def test_noalloc_plan_matches_workspace_plan_twice(cuda_lib, M, k, E):
    f = _bind(cuda_lib)
    for call in range(2):
        rng = np.random.default_rng(1000 * call + M + E)
        ids = torch.from_numpy(rng.integers(0, E, (M, k)).astype(np.int32)).cuda()
        ref = cuda_lib.hg_plan_expert_offsets(ids, E)
        st, off, s2d, d2s = _noalloc(f, ids, E)
        torch.cuda.synchronize()
        assert st == cuda_lib.HG_OK
        for got, want in zip((off, s2d, d2s), ref):
            assert torch.equal(got, want)
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def test_noalloc_plan_rejects_workspace_beyond_its_array(cuda_lib):
    f = _bind(cuda_lib)
    ids = torch.zeros((40000, 8), dtype=torch.int32, device="cuda")
    # 157 blocks x 512 experts x 4 bytes > 256 KiB
    st, *_ = _noalloc(f, ids, 512)
    assert st == cuda_lib.HG_ERR_RESOURCE
