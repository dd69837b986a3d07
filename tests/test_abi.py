"""The C-ABI library on the CPU: it builds, loads, exports every function
include/hg.h declares, and rejects bad arguments before any CUDA call.
No compute calls are made here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hg.h")
LIB = os.path.join(ROOT, "fp8_mxfp4_grouped_gb300", "libhg.so")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        from fp8_mxfp4_grouped_gb300 import build
        build.build()
    from fp8_mxfp4_grouped_gb300 import hg
    return hg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hg_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("hg_plan_expert_offsets", "hg_grouped_w4a8_gemm", "hg_get_device_status",
              "hg_plan_workspace_bytes", "hg_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\S+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        getattr(lib.lib, n)


def test_status_strings(lib):
    for code in range(8):
        s = lib.lib.hg_status_string(code)
        assert s and s != b"unknown status"
    assert lib.lib.hg_status_string(99) == b"unknown status"


def test_plan_workspace_bytes(lib):
    f = lib.hg_plan_workspace_bytes
    assert f(16, 2, 4) == 1 * 4 * 4
    assert f(16384, 8, 32) == 64 * 32 * 4
    assert f(0, 8, 32) == 4 * 32
    assert f(-1, 8, 32) == 0 and f(4, 0, 32) == 0 and f(4, 8, 0) == 0


def test_plan_block_fit(lib):
    # largest multiple of 32 <= 512 whose (warps + 2) x E x 4 bytes fit the limit
    f = lib.hg_plan_block_threads
    limit = 232448
    prev = 512
    for E in [1, 32, 512, 2048, 2880, 3072, 4608, 6144, 9216, 14000]:
        t = f(E, limit)
        assert t % 32 == 0 and 0 <= t <= 512
        assert t <= prev
        prev = t
        if t:
            assert (t // 32 + 2) * E * 4 <= limit
            if t < 512:
                assert ((t + 32) // 32 + 2) * E * 4 > limit
    assert f(32, limit) == 512
    assert f(20000, limit) == 0          # even one warp does not fit: resource error
    assert f(0, limit) == 0 and f(32, 0) == 0


def _gemm(lib, a=0x1000, asc=0x2000, w=0x4000, ws=0x8000, off=0x9000, E=4, N=256, K=512,
          rows=32, out=0xA000):
    c = ctypes.c_void_p
    return lib.lib.hg_grouped_w4a8_gemm(c(a), c(asc), c(w), c(ws), c(off), E, N, K, rows, c(out),
                                        None)


def test_gemm_argument_validation(lib):
    assert _gemm(lib, E=0) == lib.HG_ERR_INVALID_ARG
    assert _gemm(lib, rows=-1) == lib.HG_ERR_INVALID_ARG
    assert _gemm(lib, w=0) == lib.HG_ERR_INVALID_ARG
    assert _gemm(lib, off=0) == lib.HG_ERR_INVALID_ARG
    assert _gemm(lib, a=0) == lib.HG_ERR_INVALID_ARG
    assert _gemm(lib, N=200) == lib.HG_ERR_UNSUPPORTED_SHAPE
    assert _gemm(lib, K=320) == lib.HG_ERR_UNSUPPORTED_SHAPE    # K % 128 != 0
    assert _gemm(lib, K=64) == lib.HG_ERR_UNSUPPORTED_SHAPE
    assert lib.hg_gemm_ctas(4, 256, 320, 32) == 0                # rejected before any device query
    assert _gemm(lib, E=5000) == lib.HG_ERR_UNSUPPORTED_SHAPE
    assert _gemm(lib, E=513) == lib.HG_ERR_UNSUPPORTED_SHAPE   # 512 experts at most
    assert _gemm(lib, w=0x4010) == lib.HG_ERR_INVALID_ARG      # W needs 32-byte alignment
    assert _gemm(lib, a=0x1008) == lib.HG_ERR_INVALID_ARG      # A needs 16-byte alignment
    assert _gemm(lib, ws=0x8001) == lib.HG_ERR_INVALID_ARG
    # rows == 0 is a valid no-op that touches nothing
    assert _gemm(lib, rows=0, a=0, asc=0, out=0) == lib.HG_OK


def test_plan_argument_validation(lib):
    c = ctypes.c_void_p
    f = lib.lib.hg_plan_expert_offsets
    assert f(c(0x1000), -1, 8, 32, c(0x2000), c(0x3000), c(0x4000), c(0x5000), 1 << 20, None) == lib.HG_ERR_INVALID_ARG
    assert f(c(0x1000), 4, 0, 32, c(0x2000), c(0x3000), c(0x4000), c(0x5000), 1 << 20, None) == lib.HG_ERR_INVALID_ARG
    assert f(c(0x1000), 4, 8, 32, None, c(0x3000), c(0x4000), c(0x5000), 1 << 20, None) == lib.HG_ERR_INVALID_ARG
    assert f(c(0x1000), 4, 8, 32, c(0x2000), c(0x3000), c(0x4000), c(0x5000), 4, None) == lib.HG_ERR_INVALID_ARG
    assert f(None, 4, 8, 32, c(0x2000), c(0x3000), c(0x4000), c(0x5000), 1 << 20, None) == lib.HG_ERR_INVALID_ARG


def test_quantize_scatter_argument_validation(lib):
    c = ctypes.c_void_p
    f = lib.lib.hg_quantize_scatter_acts
    ok = dict(x=0x1000, M=4, K=256, k=2, d2s=0x2000, a=0x3000, s=0x4000)
    def call(**kw):
        a = dict(ok, **kw)
        return f(c(a["x"]), a["M"], a["K"], a["k"], c(a["d2s"]), c(a["a"]), c(a["s"]), None)
    assert call(M=-1) == lib.HG_ERR_INVALID_ARG
    assert call(k=0) == lib.HG_ERR_INVALID_ARG
    assert call(K=200) == lib.HG_ERR_UNSUPPORTED_SHAPE
    assert call(k=65) == lib.HG_ERR_UNSUPPORTED_SHAPE              # top_k <= 64
    assert call(x=0) == lib.HG_ERR_INVALID_ARG
    assert call(d2s=0) == lib.HG_ERR_INVALID_ARG
    assert call(x=0x1008) == lib.HG_ERR_INVALID_ARG                # 16-byte alignment
    assert call(a=0x3008) == lib.HG_ERR_INVALID_ARG
    assert call(M=0, x=0, d2s=0, a=0, s=0) == lib.HG_OK            # empty: a no-op


def test_gemm_host_workspace_bytes(lib):
    f = lib.hg_gemm_host_workspace_bytes
    # regions (each rounded up to 256 bytes): ids R*4, offsets (E+1)*4,
    # sorted_to_src R*4, src_to_sorted R*4, plan workspace, A R*K,
    # scales R*K/128, out R*N*2
    R, E, N, K = 32, 4, 256, 512
    assert lib.hg_plan_workspace_bytes(16, 2, E) == 16
    assert f(16, 2, E, N, K) == 256 * 6 + R * K + R * N * 2
    assert f(0, 8, 32, 4096, 6144) == 256 + 256          # offsets and the plan's counts
    big = f(16384, 8, 32, 4096, 6144)
    R = 16384 * 8
    assert big >= R * (4 * 3 + 6144 + 48 + 4096 * 2) and big % 256 == 0
    assert f(-1, 8, 32, 256, 512) == 0 and f(4, 0, 32, 256, 512) == 0
    assert f(4, 8, 0, 256, 512) == 0 and f(4, 8, 32, 0, 512) == 0 and f(4, 8, 32, 256, 64) == 0


def test_gemm_host_argument_validation(lib):
    c = ctypes.c_void_p
    f = lib.lib.hg_grouped_w4a8_gemm_host
    need = lib.hg_gemm_host_workspace_bytes(4, 8, 32, 256, 512)
    ok = dict(ids=0x1000, a=0x2000, s=0x3000, w=0x4000, ws_=0x5000, M=4, k=8, E=32, N=256, K=512,
              out=0x6000, off=0x7000, s2s=0x8000, wk=0x10000, wkb=need)
    def call(**kw):
        a = dict(ok, **kw)
        return f(c(a["ids"]), c(a["a"]), c(a["s"]), c(a["w"]), c(a["ws_"]), a["M"], a["k"], a["E"],
                 a["N"], a["K"], c(a["out"]), c(a["off"]), c(a["s2s"]), c(a["wk"]), a["wkb"], None)
    assert call(M=-1) == lib.HG_ERR_INVALID_ARG
    assert call(k=0) == lib.HG_ERR_INVALID_ARG
    assert call(E=0) == lib.HG_ERR_INVALID_ARG
    assert call(E=513) == lib.HG_ERR_UNSUPPORTED_SHAPE
    assert call(N=200) == lib.HG_ERR_UNSUPPORTED_SHAPE
    assert call(K=320) == lib.HG_ERR_UNSUPPORTED_SHAPE
    assert call(M=1 << 30) == lib.HG_ERR_UNSUPPORTED_SHAPE      # M*top_k >= 2^31
    assert call(w=0x4010) == lib.HG_ERR_INVALID_ARG              # W needs 32-byte alignment
    assert call(ws_=0x5001) == lib.HG_ERR_INVALID_ARG
    assert call(ids=0) == lib.HG_ERR_INVALID_ARG
    assert call(a=0) == lib.HG_ERR_INVALID_ARG
    assert call(out=0) == lib.HG_ERR_INVALID_ARG
    assert call(wk=0) == lib.HG_ERR_INVALID_ARG
    assert call(wk=0x10010) == lib.HG_ERR_INVALID_ARG            # workspace 256-byte aligned
    assert call(wkb=need - 1) == lib.HG_ERR_INVALID_ARG


def test_plan_launches_rejects_bad_arguments_without_a_device(lib):
    # argument checks come first; sizes that need the device's limits read -1
    # here only when no device can be queried
    assert lib.hg_plan_launches(-1, 8, 32) == -1
    assert lib.hg_plan_launches(4, 0, 32) == -1
    assert lib.hg_plan_launches(4, 8, 0) == -1
    assert lib.hg_plan_launches(0, 8, 32) == 0
    assert lib.hg_plan_launches(1 << 30, 8, 32) == -1


def test_shutdown_without_a_device(lib):
    # host-only: drops the caches, nothing to free, safe to repeat
    assert lib.lib.hg_shutdown() == lib.HG_OK
    assert lib.lib.hg_shutdown() == lib.HG_OK
