"""Python binding of libhg (the C ABI in include/hg.h).

Argument marshalling only: every step of the computation runs in the
library's CUDA kernels.  Tensors are torch CUDA tensors (device memory and
streams only); their data pointers are passed straight through ctypes.
There is no fallback: if the library is missing, importing this module
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libhg.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with "
                      "`python -m fp8_mxfp4_grouped_gb300.build` (nvcc, sm_103a)")

lib = ctypes.CDLL(LIB_PATH)

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_u32 = ctypes.c_uint32
_sz = ctypes.c_size_t

lib.hg_status_string.argtypes = [ctypes.c_int]
lib.hg_status_string.restype = ctypes.c_char_p
lib.hg_version.argtypes = []
lib.hg_version.restype = ctypes.c_int
lib.hg_shutdown.argtypes = []
lib.hg_shutdown.restype = ctypes.c_int
lib.hg_plan_workspace_bytes.argtypes = [_i32, _i32, _i32]
lib.hg_plan_workspace_bytes.restype = _sz
lib.hg_plan_block_threads.argtypes = [_i32, _i32]
lib.hg_plan_block_threads.restype = _i32
lib.hg_plan_launches.argtypes = [_i32, _i32, _i32]
lib.hg_plan_launches.restype = _i32
lib.hg_plan_expert_offsets.argtypes = [_p, _i32, _i32, _i32, _p, _p, _p, _p, _sz, _p]
lib.hg_plan_expert_offsets.restype = ctypes.c_int
lib.hg_grouped_w4a8_gemm.argtypes = [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _p, _p]
lib.hg_grouped_w4a8_gemm.restype = ctypes.c_int
lib.hg_grouped_w4a8_gemm_mmajor.argtypes = [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _p, _p]
lib.hg_grouped_w4a8_gemm_mmajor.restype = ctypes.c_int
lib.hg_quantize_gather_acts.argtypes = [_p, _i32, _i32, _i32, _p, _p, _p, _p]
lib.hg_quantize_gather_acts.restype = ctypes.c_int
lib.hg_quantize_scatter_acts.argtypes = [_p, _i32, _i32, _i32, _p, _p, _p, _p]
lib.hg_quantize_scatter_acts.restype = ctypes.c_int
lib.hg_combine_topk.argtypes = [_p, _p, _p, _i32, _i32, _i32, _p, _p]
lib.hg_combine_topk.restype = ctypes.c_int
lib.hg_get_device_status.argtypes = [_p, ctypes.POINTER(_u32)]
lib.hg_get_device_status.restype = ctypes.c_int
lib.hg_selftest_wait_timeout.argtypes = [_u32, _p]
lib.hg_selftest_wait_timeout.restype = ctypes.c_int
lib.hg_set_wait_timeout_us.argtypes = [_u32]
lib.hg_set_wait_timeout_us.restype = None
lib.hg_gemm_token_tile.argtypes = [_i32, _i32, _i32, _i32]
lib.hg_gemm_token_tile.restype = _i32
lib.hg_gemm_ctas.argtypes = [_i32, _i32, _i32, _i32]
lib.hg_gemm_ctas.restype = _i32
lib.hg_set_gemm_variant.argtypes = [_i32]
lib.hg_set_gemm_variant.restype = _i32
lib.hg_gemm_host_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32]
lib.hg_gemm_host_workspace_bytes.restype = _sz
lib.hg_grouped_w4a8_gemm_host.argtypes = [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _p,
                                          _p, _p, _p, _sz, _p]
lib.hg_grouped_w4a8_gemm_host.restype = ctypes.c_int

HG_OK = 0
HG_ERR_INVALID_ARG = 1
HG_ERR_UNSUPPORTED_SHAPE = 2
HG_ERR_RESOURCE = 3
HG_ERR_CUDA = 4
HG_ERR_TIMEOUT = 5
HG_ERR_BAD_OFFSETS = 6
HG_ERR_BAD_IDS = 7


class HgError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {lib.hg_status_string(status).decode()} ({status})")


def _check(status: int, what: str):
    if status != HG_OK:
        raise HgError(status, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def hg_shutdown() -> None:
    """Drop the library's per-device caches (see include/hg.h)."""
    _check(lib.hg_shutdown(), "hg_shutdown")


def hg_plan_workspace_bytes(M: int, top_k: int, E: int) -> int:
    return int(lib.hg_plan_workspace_bytes(M, top_k, E))


def hg_plan_block_threads(E: int, smem_limit_bytes: int) -> int:
    return int(lib.hg_plan_block_threads(E, smem_limit_bytes))


def hg_plan_launches(M: int, top_k: int, E: int) -> int:
    return int(lib.hg_plan_launches(M, top_k, E))


def hg_plan_expert_offsets(topk_ids: torch.Tensor, E: int, expert_offsets=None,
                           sorted_to_src=None, src_to_sorted=None, workspace=None,
                           stream=None):
    """Routing plan on the GPU. Returns (expert_offsets, sorted_to_src, src_to_sorted)."""
    assert topk_ids.dtype == torch.int32 and topk_ids.is_contiguous() and topk_ids.dim() == 2
    M, k = topk_ids.shape
    dev = topk_ids.device
    R = M * k
    if expert_offsets is None:
        expert_offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if sorted_to_src is None:
        sorted_to_src = torch.empty(R, dtype=torch.int32, device=dev)
    if src_to_sorted is None:
        src_to_sorted = torch.empty(R, dtype=torch.int32, device=dev)
    need = hg_plan_workspace_bytes(M, k, E)
    if workspace is None:
        workspace = torch.empty(max(need, 4), dtype=torch.uint8, device=dev)
    st = lib.hg_plan_expert_offsets(_ptr(topk_ids), M, k, E, _ptr(expert_offsets),
                                    _ptr(sorted_to_src), _ptr(src_to_sorted), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "hg_plan_expert_offsets")
    return expert_offsets, sorted_to_src, src_to_sorted


def hg_grouped_w4a8_gemm(a_fp8: torch.Tensor, a_scale: torch.Tensor, w_fp4: torch.Tensor,
                         w_scale: torch.Tensor, expert_offsets: torch.Tensor, out=None,
                         stream=None) -> torch.Tensor:
    """Grouped-contiguous W4A8 GEMM. Returns out [rows, N] as torch.bfloat16."""
    E, N, K2 = w_fp4.shape
    K = 2 * K2
    rows = a_fp8.shape[0]
    for t in (a_fp8, a_scale, w_fp4, w_scale, expert_offsets):
        assert t.is_contiguous()
    assert a_fp8.shape == (rows, K) and a_scale.shape == (rows, K // 128)
    assert w_scale.shape == (E, N, K // 32) and expert_offsets.numel() == E + 1
    if out is None:
        out = torch.empty((rows, N), dtype=torch.bfloat16, device=a_fp8.device)
    st = lib.hg_grouped_w4a8_gemm(_ptr(a_fp8), _ptr(a_scale), _ptr(w_fp4), _ptr(w_scale),
                                  _ptr(expert_offsets), E, N, K, rows, _ptr(out),
                                  _stream(stream))
    _check(st, "hg_grouped_w4a8_gemm")
    return out


def hg_gemm_host_workspace_bytes(M: int, top_k: int, E: int, N: int, K: int) -> int:
    return int(lib.hg_gemm_host_workspace_bytes(M, top_k, E, N, K))


def hg_grouped_w4a8_gemm_host(topk_ids: torch.Tensor, a_fp8: torch.Tensor, a_scale: torch.Tensor,
                              w_fp4: torch.Tensor, w_scale: torch.Tensor, E: int,
                              out: torch.Tensor, workspace: torch.Tensor,
                              expert_offsets=None, sorted_to_src=None, stream=None):
    """Plan + GEMM from host buffers (CPU tensors, page-locked for asynchronous
    copies): topk_ids int32 [M, top_k], a_fp8 uint8 [M*top_k, K] in the plan's
    order, a_scale uint8 [M*top_k, K/128], out bfloat16 [M*top_k, N]; optional
    host outputs expert_offsets int32 [E+1] and sorted_to_src int32 [M*top_k].
    Weights and workspace (uint8, hg_gemm_host_workspace_bytes) are on the
    device.  Asynchronous on `stream`: the host outputs are valid once the
    stream has reached the end of the call."""
    M, k = topk_ids.shape
    R = M * k
    _, N, K2 = w_fp4.shape
    K = 2 * K2
    for t in (topk_ids, a_fp8, a_scale, out):
        assert not t.is_cuda and t.is_contiguous()
    for t in (expert_offsets, sorted_to_src):
        assert t is None or (not t.is_cuda and t.is_contiguous())
    assert topk_ids.dtype == torch.int32
    assert a_fp8.shape == (R, K) and a_scale.shape == (R, K // 128) and out.shape == (R, N)
    assert expert_offsets is None or expert_offsets.numel() == E + 1
    assert sorted_to_src is None or sorted_to_src.numel() == R
    assert workspace.is_cuda and workspace.dtype == torch.uint8
    st = lib.hg_grouped_w4a8_gemm_host(_ptr(topk_ids), _ptr(a_fp8), _ptr(a_scale), _ptr(w_fp4),
                                       _ptr(w_scale), M, k, E, N, K, _ptr(out),
                                       _ptr(expert_offsets), _ptr(sorted_to_src), _ptr(workspace),
                                       workspace.numel(), _stream(stream))
    _check(st, "hg_grouped_w4a8_gemm_host")
    return out


def hg_grouped_w4a8_gemm_mmajor(a_fp8: torch.Tensor, a_scale_mmajor: torch.Tensor,
                                w_fp4: torch.Tensor, w_scale: torch.Tensor,
                                expert_offsets: torch.Tensor, out=None, stream=None) -> torch.Tensor:
    """The GEMM with activation scales laid out [K/128, rows]. Returns out [rows, N] bf16."""
    E, N, K2 = w_fp4.shape
    K = 2 * K2
    rows = a_fp8.shape[0]
    for t in (a_fp8, a_scale_mmajor, w_fp4, w_scale, expert_offsets):
        assert t.is_contiguous()
    assert a_fp8.shape == (rows, K) and a_scale_mmajor.shape == (K // 128, rows)
    assert w_scale.shape == (E, N, K // 32) and expert_offsets.numel() == E + 1
    if out is None:
        out = torch.empty((rows, N), dtype=torch.bfloat16, device=a_fp8.device)
    st = lib.hg_grouped_w4a8_gemm_mmajor(_ptr(a_fp8), _ptr(a_scale_mmajor), _ptr(w_fp4),
                                         _ptr(w_scale), _ptr(expert_offsets), E, N, K, rows,
                                         _ptr(out), _stream(stream))
    _check(st, "hg_grouped_w4a8_gemm_mmajor")
    return out


def hg_quantize_gather_acts(x_bf16: torch.Tensor, top_k: int, sorted_to_src: torch.Tensor,
                            a_fp8=None, a_scale=None, stream=None):
    """BF16 [M, K] tokens -> (E4M3 [M*top_k, K], E8M0 [M*top_k, K/128]) in sorted order."""
    assert x_bf16.dtype == torch.bfloat16 and x_bf16.is_contiguous() and x_bf16.dim() == 2
    M, K = x_bf16.shape
    R = M * top_k
    if a_fp8 is None:
        a_fp8 = torch.empty((R, K), dtype=torch.uint8, device=x_bf16.device)
    if a_scale is None:
        a_scale = torch.empty((R, K // 128), dtype=torch.uint8, device=x_bf16.device)
    st = lib.hg_quantize_gather_acts(_ptr(x_bf16), M, K, top_k, _ptr(sorted_to_src), _ptr(a_fp8),
                                     _ptr(a_scale), _stream(stream))
    _check(st, "hg_quantize_gather_acts")
    return a_fp8, a_scale


def hg_quantize_scatter_acts(x_bf16: torch.Tensor, top_k: int, src_to_sorted: torch.Tensor,
                             a_fp8=None, a_scale=None, stream=None):
    """BF16 [M, K] tokens -> (E4M3 [M*top_k, K], E8M0 [M*top_k, K/128]); token t's codes
    go to rows src_to_sorted[t*top_k + j]."""
    assert x_bf16.dtype == torch.bfloat16 and x_bf16.is_contiguous() and x_bf16.dim() == 2
    M, K = x_bf16.shape
    R = M * top_k
    if a_fp8 is None:
        a_fp8 = torch.empty((R, K), dtype=torch.uint8, device=x_bf16.device)
    if a_scale is None:
        a_scale = torch.empty((R, K // 128), dtype=torch.uint8, device=x_bf16.device)
    st = lib.hg_quantize_scatter_acts(_ptr(x_bf16), M, K, top_k, _ptr(src_to_sorted),
                                      _ptr(a_fp8), _ptr(a_scale), _stream(stream))
    _check(st, "hg_quantize_scatter_acts")
    return a_fp8, a_scale


def hg_combine_topk(y_bf16: torch.Tensor, src_to_sorted: torch.Tensor, topk_weights: torch.Tensor,
                    out=None, stream=None) -> torch.Tensor:
    """out[t] = sum_j w[t, j] * y[src_to_sorted[t*k + j]]  (FP32 sum, BF16 result)."""
    M, k = topk_weights.shape
    N = y_bf16.shape[1]
    assert topk_weights.dtype == torch.float32 and topk_weights.is_contiguous()
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=y_bf16.device)
    st = lib.hg_combine_topk(_ptr(y_bf16), _ptr(src_to_sorted), _ptr(topk_weights), M, k, N,
                             _ptr(out), _stream(stream))
    _check(st, "hg_combine_topk")
    return out


def hg_get_device_status(stream=None):
    """(status, detail) of the device status word; synchronises the stream."""
    detail = _u32(0)
    st = lib.hg_get_device_status(_stream(stream), ctypes.byref(detail))
    return int(st), int(detail.value)


def hg_selftest_wait_timeout(timeout_us: int, stream=None):
    _check(lib.hg_selftest_wait_timeout(timeout_us, _stream(stream)), "hg_selftest_wait_timeout")


def hg_set_wait_timeout_us(timeout_us: int):
    lib.hg_set_wait_timeout_us(timeout_us)


def hg_gemm_token_tile(E: int, N: int, K: int, rows: int) -> int:
    return int(lib.hg_gemm_token_tile(E, N, K, rows))


def hg_gemm_ctas(E: int, N: int, K: int, rows: int) -> int:
    return int(lib.hg_gemm_ctas(E, N, K, rows))


def hg_set_gemm_variant(variant: int) -> int:
    prev = int(lib.hg_set_gemm_variant(variant))
    if prev < 0:
        raise ValueError(f"invalid GEMM variant {variant}")
    return prev
