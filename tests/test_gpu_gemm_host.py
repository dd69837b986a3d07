"""hg_grouped_w4a8_gemm_host: the routing plan and the GEMM called on host
buffers.  Its results equal those of the two device calls bit for bit (the
same kernels on the same bytes), and the small case also matches the oracle
element by element."""
import numpy as np
import pytest
import torch

from oracle import gemm as G
from oracle.plan import plan_expert_offsets
from synth import make_case
from tests.gpu_util import assert_rows_close, bf16_bits, np_u8

pytestmark = pytest.mark.gpu


def _pinned(t):
    return t.contiguous().pin_memory()


def _host_call(hg, c, with_plan_outputs=True, stream=None):
    R = c.M * c.top_k
    ids = _pinned(torch.from_numpy(np.ascontiguousarray(c.topk_ids)))
    a = _pinned(c.a_fp8.cpu())
    a_s = _pinned(c.a_scale.cpu())
    out = torch.empty((R, c.N), dtype=torch.bfloat16).pin_memory()
    off = torch.empty(c.E + 1, dtype=torch.int32).pin_memory() if with_plan_outputs else None
    s2s = torch.empty(R, dtype=torch.int32).pin_memory() if with_plan_outputs else None
    ws = torch.empty(hg.hg_gemm_host_workspace_bytes(c.M, c.top_k, c.E, c.N, c.K),
                     dtype=torch.uint8, device="cuda")
    hg.hg_grouped_w4a8_gemm_host(ids, a, a_s, c.w_fp4.cuda(), c.w_scale.cuda(), c.E, out, ws,
                                 expert_offsets=off, sorted_to_src=s2s, stream=stream)
    torch.cuda.synchronize()
    return out, off, s2s


def _device_calls(hg, c):
    off, s2s, _ = hg.hg_plan_expert_offsets(torch.from_numpy(c.topk_ids).cuda(), c.E)
    out = hg.hg_grouped_w4a8_gemm(c.a_fp8.cuda(), c.a_scale.cuda(), c.w_fp4.cuda(),
                                  c.w_scale.cuda(), off)
    torch.cuda.synchronize()
    return out.cpu(), off.cpu(), s2s.cpu()


def test_tiny_case_matches_oracle(cuda_lib):
    c = make_case(0, 16)
    out, off, s2s = _host_call(cuda_lib, c)
    ref_off, ref_s2s, _, n_invalid = plan_expert_offsets(c.topk_ids, c.E)
    assert n_invalid == 0
    assert np.array_equal(off.numpy(), ref_off)
    assert np.array_equal(s2s.numpy(), ref_s2s)
    ref = G.grouped_w4a8_gemm(np_u8(c.a_fp8), np_u8(c.a_scale), np_u8(c.w_fp4), np_u8(c.w_scale),
                              ref_off, c.E, c.N, c.K)
    assert_rows_close(bf16_bits(out), ref, "host-buffer call, config 0")
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


@pytest.mark.parametrize("cid,M,proj,routing", [
    (1, 64, "gate_up", "biased"),      # few rows per expert, some experts empty
    (2, 512, "down", "biased"),
    (3, 8, "w13", "uniform"),          # the split-K shape
    (4, 4096, "down", "uniform"),      # full size, the 224-row shape
])
def test_equals_device_calls(cuda_lib, cid, M, proj, routing):
    c = make_case(cid, M, projection=proj, routing=routing)
    out_h, off_h, s2s_h = _host_call(cuda_lib, c, stream=torch.cuda.Stream())
    out_d, off_d, s2s_d = _device_calls(cuda_lib, c)
    assert torch.equal(off_h, off_d) and torch.equal(s2s_h, s2s_d)
    assert torch.equal(out_h.view(torch.int16), out_d.view(torch.int16))
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def test_optional_outputs_and_empty_batch(cuda_lib):
    c = make_case(1, 64, projection="gate_up", routing="biased")
    out, off, s2s = _host_call(cuda_lib, c, with_plan_outputs=False)
    assert off is None and s2s is None
    out_d, _, _ = _device_calls(cuda_lib, c)
    assert torch.equal(out.view(torch.int16), out_d.view(torch.int16))
    # M = 0: nothing to copy but the (zero) offsets
    E, N, K = c.E, c.N, c.K
    ws = torch.empty(cuda_lib.hg_gemm_host_workspace_bytes(0, 8, E, N, K), dtype=torch.uint8,
                     device="cuda")
    off0 = torch.full((E + 1,), -7, dtype=torch.int32).pin_memory()
    empty_ids = torch.empty((0, 8), dtype=torch.int32)
    cuda_lib.hg_grouped_w4a8_gemm_host(empty_ids, torch.empty((0, K), dtype=torch.uint8),
                                       torch.empty((0, K // 128), dtype=torch.uint8),
                                       c.w_fp4.cuda(), c.w_scale.cuda(), E,
                                       torch.empty((0, N), dtype=torch.bfloat16), ws,
                                       expert_offsets=off0)
    torch.cuda.synchronize()
    assert torch.equal(off0, torch.zeros(E + 1, dtype=torch.int32))


def test_pageable_host_buffers(cuda_lib):
    # not page-locked: the copies are staged by the driver, the results are the same
    c = make_case(2, 64, projection="down", routing="biased")
    R = c.M * c.top_k
    out = torch.empty((R, c.N), dtype=torch.bfloat16)
    ws = torch.empty(cuda_lib.hg_gemm_host_workspace_bytes(c.M, c.top_k, c.E, c.N, c.K),
                     dtype=torch.uint8, device="cuda")
    cuda_lib.hg_grouped_w4a8_gemm_host(torch.from_numpy(np.ascontiguousarray(c.topk_ids)),
                                       c.a_fp8.cpu().contiguous(), c.a_scale.cpu().contiguous(),
                                       c.w_fp4.cuda(), c.w_scale.cuda(), c.E, out, ws)
    torch.cuda.synchronize()
    out_d, _, _ = _device_calls(cuda_lib, c)
    assert torch.equal(out.view(torch.int16), out_d.view(torch.int16))


def test_graph_capture_and_replay(cuda_lib):
    # the whole host-buffer call captured once; replays read the pinned inputs
    # as they are at replay time and write the pinned output
    c1 = make_case(1, 64, projection="gate_up", routing="biased")
    c2 = make_case(1, 64, projection="gate_up", routing="uniform")
    R = c1.M * c1.top_k
    ids = _pinned(torch.from_numpy(np.ascontiguousarray(c1.topk_ids)))
    a = _pinned(c1.a_fp8.cpu())
    a_s = _pinned(c1.a_scale.cpu())
    out = torch.empty((R, c1.N), dtype=torch.bfloat16).pin_memory()
    ws = torch.empty(cuda_lib.hg_gemm_host_workspace_bytes(c1.M, c1.top_k, c1.E, c1.N, c1.K),
                     dtype=torch.uint8, device="cuda")
    w, w_s = c1.w_fp4.cuda(), c1.w_scale.cuda()
    s = torch.cuda.Stream()
    cuda_lib.hg_grouped_w4a8_gemm_host(ids, a, a_s, w, w_s, c1.E, out, ws, stream=s)   # warm-up
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        cuda_lib.hg_grouped_w4a8_gemm_host(ids, a, a_s, w, w_s, c1.E, out, ws,
                                           stream=torch.cuda.current_stream())
    for c in (c2, c1):
        ids.copy_(torch.from_numpy(np.ascontiguousarray(c.topk_ids)))
        a.copy_(c.a_fp8.cpu())
        a_s.copy_(c.a_scale.cpu())
        g.replay()
        torch.cuda.synchronize()
        out_d, _, _ = _device_calls(cuda_lib, c)
        assert torch.equal(out.view(torch.int16), out_d.view(torch.int16))
    assert cuda_lib.hg_get_device_status()[0] == cuda_lib.HG_OK


def test_dropped_ids(cuda_lib):
    # ids outside [0, E) are dropped by the plan: the rows before off[E] carry
    # results equal to the device calls', the count is reported
    c = make_case(1, 64, projection="gate_up", routing="biased")
    ids = np.ascontiguousarray(c.topk_ids).copy()
    ids[::7, 0] = -1
    ids[3::11, 1] = c.E
    c.topk_ids = ids
    cuda_lib.hg_get_device_status()
    out_h, off_h, s2s_h = _host_call(cuda_lib, c)
    st, detail = cuda_lib.hg_get_device_status()
    ref_off, ref_s2s, _, bad = plan_expert_offsets(ids, c.E)
    assert bad > 0 and st == cuda_lib.HG_ERR_BAD_IDS and detail == bad
    assert np.array_equal(off_h.numpy(), ref_off) and np.array_equal(s2s_h.numpy(), ref_s2s)
    out_d, off_d, _ = _device_calls(cuda_lib, c)
    cuda_lib.hg_get_device_status()
    n = int(ref_off[-1])
    assert torch.equal(out_h[:n].view(torch.int16), out_d[:n].view(torch.int16))
