#!/usr/bin/env python3
"""Benchmark of the grouped FP8 x MXFP4 MoE GEMM hot path (routing plan + GEMM).

Workload (default): the gate/up projection of the pages' headline table --
E=32 experts, top-8, N=4096, K=6144, unbalanced (biased) routing -- swept over
M in {64, 256, 512, 768, 1152, 1536, 2048} tokens.  One step = for every M:
an L2 flush (a write of 2x the L2 size, then a read of another 2x, so that
the flush's own write-backs are not charged to the timed kernels), then the
routing plan and the grouped GEMM in one CUDA-event bracket on the launching
stream (the GEMM is launched with programmatic dependent launch, so its
prologue overlaps the plan).  An untimed pass afterwards splits each M into
plan alone, plan + GEMM and GEMM alone for the per-shape report.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints ONE JSON line (rank 0).  value = total GEMM FLOPs of the sweep /
device time of the plan + GEMM brackets (TFLOP/s, whole job).  The reference arm
(--impl reference) times the CPU oracle on a bounded sample of the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "grouped FP8×MXFP4 MoE GEMM µs & TFLOP/s vs tokens M; % of roofline"
UNIT = "TFLOP/s"
CONFIG_ID = 1
WORKLOAD = "gate_up E=32 top8 N=4096 K=6144 unbalanced, M sweep 64..2048"
FP8_OVER_BF16 = 2.0   # nominal dense fp8 / bf16 tensor ratio


class L2Flush:
    """Cold L2 before a timed launch: write a buffer of 2x the L2 size, then
    read a second one of the same size.  The read evicts the dirty lines the
    write left, so their write-backs happen here, untimed, and not inside the
    kernel that follows."""

    DESCRIPTION = ("flushed before every timed bracket (plan + GEMM): 2x L2 written, then another 2x L2 read "
                   "(write-backs of the flush land before the timed region)")

    def __init__(self, l2_bytes, dev):
        import torch
        self.w = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev)
        self.r = torch.zeros(2 * l2_bytes // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self, v):
        self.w.fill_(int(v) & 0xFF)
        self.sink.copy_(self.r.sum())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm_gbs=d["hbm_gbs"], bf16=d["bf16_tflops"],
                    bf16_sust=d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                    source="measured")
    return dict(hbm_gbs=6800.0, bf16=1900.0, bf16_sust=1700.0, source="fallback")


def measured_traffic(M):
    """ncu DRAM bytes per launch of the GEMM at this M, from the committed profile
    summary -- only while the kernel source still hashes to the captured version."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", f"grouped_w4a8_gemm_gate_up_M{M}.md")
    src = os.path.join(ROOT, "fp8_mxfp4_grouped_gb300", "csrc", "gemm.cu")
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    fields = {}
    for line in open(prof):
        if ":" in line and not line.startswith(("|", "#", " ")):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if fields.get("kernel_source_sha256_16") != sha or "dram_bytes_per_launch" not in fields:
        return None
    return float(fields["dram_bytes_per_launch"])


def host_link_gbs(cs, dev):
    """Host<->device copy rates (GB/s) of this box with the largest batch's
    pinned buffers: upload alone, download alone, and both at once (total);
    each the best of five timed copies."""
    h = cs["host"]
    up_d = torch.empty_like(h["a"], device=dev)
    dn_d = torch.empty_like(h["out"], device=dev)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()

    def timed(fn, reps=5):
        # best of single timed copies: an occasional slow one (see the
        # end-to-end leg) must not lower the rate
        fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize()
            best = min(best, time.perf_counter() - t0)
        return best

    def up():
        with torch.cuda.stream(s1):
            up_d.copy_(h["a"], non_blocking=True)

    def down():
        with torch.cuda.stream(s2):
            h["out"].copy_(dn_d, non_blocking=True)

    nu, nd = h["a"].numel(), h["out"].numel() * 2
    tu, td = timed(up), timed(down)
    tb = timed(lambda: (up(), down()))
    return dict(h2d=round(nu / tu / 1e9, 1), d2h=round(nd / td / 1e9, 1),
                both=round((nu + nd) / tb / 1e9, 1))


def device_buffers(c, dev, hg):
    """Device-side ids, plan outputs, plan workspace and GEMM output of one case."""
    R = c.R
    return dict(
        ids=torch.from_numpy(c.topk_ids).to(dev),
        off=torch.empty(c.E + 1, dtype=torch.int32, device=dev),
        s2d=torch.empty(R, dtype=torch.int32, device=dev),
        d2s=torch.empty(R, dtype=torch.int32, device=dev),
        ws=torch.empty(max(4, hg.hg_plan_workspace_bytes(c.M, c.top_k, c.E)),
                       dtype=torch.uint8, device=dev),
        out=torch.empty((R, c.N), dtype=torch.bfloat16, device=dev),
    )


def active_experts(bufs, c, stream, hg):
    """Experts with at least one row, counted from the GPU plan's offsets
    (untimed bookkeeping for the roofline's weight bytes)."""
    hg.hg_plan_expert_offsets(bufs["ids"], c.E, bufs["off"], bufs["s2d"], bufs["d2s"], bufs["ws"],
                              stream=stream)
    stream.synchronize()
    return int(np.count_nonzero(np.diff(bufs["off"].cpu().numpy())))


def sweep_entry(cs, pg_us, p_us, ga_us, peaks, fp8_peak):
    """One shape against its roofline.  pg_us: plan + GEMM in one event bracket
    (the GEMM launched right behind the plan with programmatic dependent
    launch); p_us: the plan alone; ga_us: the GEMM alone in its own bracket.
    gemm_us = pg_us - p_us, the GEMM's time in the plan -> GEMM sequence;
    roof_frac = max(HBM time, FP8 tensor time) / gemm_us; hbm_frac = algorithmic
    bytes / gemm_us / HBM peak; the *_alone fractions use ga_us."""
    t_hbm = cs["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = cs["flops"] / (fp8_peak * 1e12)
    g_us = pg_us - p_us
    return dict(M=cs["M"], R=cs["R"], E_act=cs["e_act"], gemm_us=round(g_us, 2),
                plan_us=round(p_us, 2), plan_gemm_us=round(pg_us, 2),
                gemm_alone_us=round(ga_us, 2),
                tflops=round(cs["flops"] / g_us / 1e6, 1),
                gbs=round(cs["bytes"] / g_us / 1e3, 1),
                bound="hbm" if t_hbm >= t_tc else "tensor",
                roof_frac=round(max(t_hbm, t_tc) / (g_us * 1e-6), 3),
                hbm_frac=round(t_hbm / (g_us * 1e-6), 3),
                roof_frac_alone=round(max(t_hbm, t_tc) / (ga_us * 1e-6), 3),
                hbm_frac_alone=round(t_hbm / (ga_us * 1e-6), 3))


def time_breakdown(flush, stream, hg, c, b, reps, warm=3):
    """Median device time of the plan alone, plan + GEMM in one bracket, and the
    GEMM alone (each after its own L2 flush)."""
    plan = lambda: hg.hg_plan_expert_offsets(b["ids"], c.E, b["off"], b["s2d"], b["d2s"],
                                             b["ws"], stream=stream)
    gemm = lambda: hg.hg_grouped_w4a8_gemm(c.a_fp8, c.a_scale, c.w_fp4, c.w_scale, b["off"],
                                           out=b["out"], stream=stream)
    ev = {"p": [], "pg": [], "g": []}
    for it in range(warm + reps):
        for key, fns in (("p", (plan,)), ("pg", (plan, gemm)), ("g", (gemm,))):
            with torch.cuda.stream(stream):
                flush(it)
                e = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
                e[0].record(stream)
                for fn in fns:
                    fn()
                e[1].record(stream)
            if it >= warm:
                ev[key].append(e)
    torch.cuda.synchronize()
    med = {k: statistics.median(e[0].elapsed_time(e[1]) * 1e3 for e in v) for k, v in ev.items()}
    return med["p"], med["pg"], med["g"]


# The other workloads' shapes, each measured like the headline sweep (L2
# flushed before every bracket) and reported beside it.
OTHER_WORKLOADS = [(2, "down", "biased"), (3, "w13", "uniform"), (3, "w2", "uniform"),
                   (4, "gate_up", "uniform"), (4, "gate_up", "biased"),
                   (4, "down", "uniform"), (4, "down", "biased")]


def time_other_workloads(flush, stream, peaks, fp8_peak, hg, reps, warm=3):
    """Every M of the other workloads: plan alone, plan + GEMM in one bracket,
    GEMM alone (time_breakdown)."""
    from synth import make_case
    from synth.inputs import CONFIGS
    dev = torch.device("cuda")
    out = []
    for cid, proj, routing in OTHER_WORKLOADS:
        rows = []
        c = None
        for M in CONFIGS[cid]["Ms"]:
            c = make_case(cid, M, projection=proj, routing=routing, device=dev)
            b = device_buffers(c, dev, hg)
            e_act = active_experts(b, c, stream, hg)
            flops, byts = algorithmic(c.R, e_act, c.E, c.N, c.K)
            p, pg, ga = time_breakdown(flush, stream, hg, c, b, reps, warm)
            cs = dict(M=M, R=c.R, e_act=e_act, flops=flops, bytes=byts)
            entry = sweep_entry(cs, pg, p, ga, peaks, fp8_peak)
            entry["variant_token_tile"] = hg.hg_gemm_token_tile(c.E, c.N, c.K, c.R)
            rows.append(entry)
            del b
        out.append(dict(config=cid, projection=proj, routing=routing, E=c.E, top_k=c.top_k,
                        N=c.N, K=c.K, reps=reps, sweep=rows))
        del c
        torch.cuda.empty_cache()
    st, detail = hg.hg_get_device_status()
    if st != hg.HG_OK:
        raise RuntimeError(f"device status {st} detail {detail} after the other workloads")
    return out


def target_summary(headline_sweep, others):
    """The two throughput targets over every measured shape: the lowest roofline
    fraction at M >= 4096, and the lowest HBM-roofline fraction at M <= 256.
    Both take the GEMM's time in the plan -> GEMM sequence (gemm_us); the
    lowest fraction of the GEMM timed alone is given beside each."""
    rows = [("config1 gate_up biased", r) for r in headline_sweep]
    for w in others:
        rows += [(f"config{w['config']} {w['projection']} {w['routing']}", r) for r in w["sweep"]]
    big = [(n, r) for n, r in rows if r["M"] >= 4096]
    small = [(n, r) for n, r in rows if r["M"] <= 256]
    out = {}
    for key, sel, frac, target in (("m_ge_4096_min_roof_frac", big, "roof_frac", 0.70),
                                   ("m_le_256_min_hbm_frac", small, "hbm_frac", 0.50)):
        if not sel:
            continue
        n, r = min(sel, key=lambda x: x[1][frac])
        na, ra = min(sel, key=lambda x: x[1][frac + "_alone"])
        out[key] = dict(value=r[frac], at=f"{n} M={r['M']}", target=target,
                        timing="GEMM time in the plan -> GEMM sequence (plan + GEMM bracket "
                               "minus plan alone)",
                        below=[f"{a} M={b['M']}: {b[frac]}" for a, b in sel if b[frac] < target],
                        gemm_alone=dict(value=ra[frac + "_alone"], at=f"{na} M={ra['M']}",
                                        below=sum(b[frac + "_alone"] < target for _, b in sel)))
    return out


def algorithmic(R, E_act, E, N, K):
    """GEMM flops and the bytes each operand must cross HBM once."""
    flops = 2.0 * R * N * K
    byts = (E_act * N * K / 2 + E_act * N * K / 32 + R * K + R * K / 128 + 2.0 * R * N
            + 4.0 * (E + 1))
    return flops, byts


# ------------------------------------------------------------ distributed --

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def reduce_scalar(x: float, op: str, world: int) -> float:
    """Max or sum of a per-rank scalar over all ranks (identity for one rank)."""
    if world <= 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """SM clock and clock-event reasons of the benchmarked GPU, sampled in the
    background while timing (read-only queries).  The GPU is found by its PCI
    bus id, so the samples follow the CUDA device even when device indices are
    remapped.  NVML through ctypes polls every 50 ms; without NVML,
    nvidia-smi does every 200 ms."""

    REASONS = (("sw_power_cap", 0x4), ("hw_slowdown", 0x8), ("sw_thermal_slowdown", 0x20),
               ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80))
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0, period_s=0.05):
        self.period_s = period_s
        self.bus = None
        try:
            pr = torch.cuda.get_device_properties(index)
            self.bus = f"{pr.pci_domain_id:08X}:{pr.pci_bus_id:02X}:{pr.pci_device_id:02X}.0"
        except Exception:
            pass
        self.index = index
        self.samples = []     # (sm_mhz, reason names)
        self.max_mhz = None
        self.source = None
        self._stop = threading.Event()
        self.thread = None
        self.proc = None

    # -- NVML (libnvidia-ml, read-only calls)
    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if self.bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(
                self.bus.encode(), ctypes.byref(h)) != 0:
            return None
        get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # 1 = SM clock
            self.max_mhz = float(mx.value)
        return lib, h, get_reasons

    def _nvml_loop(self, lib, h, get_reasons):
        import ctypes
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                    get_reasons(h, ctypes.byref(rs)) == 0:
                self.samples.append((float(clk.value),
                                     [n for n, bit in self.REASONS if rs.value & bit]))
            self._stop.wait(self.period_s)
        lib.nvmlShutdown()

    # -- nvidia-smi fallback
    def _smi_loop(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm, mx = float(f[0]), float(f[1])
            except ValueError:
                continue
            self.max_mhz = mx
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            self.samples.append((sm, [n for n, v in zip(names, f[4:8])
                                      if v.lower().startswith("active")]))

    def start(self):
        try:
            opened = self._nvml_open()
        except (OSError, AttributeError):
            opened = None
        if opened is not None:
            self.source = "nvml"
            self.thread = threading.Thread(target=self._nvml_loop, args=opened, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.bus or str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.source = "nvidia-smi"
            self.thread = threading.Thread(target=self._smi_loop, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.source is None:
            return None
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)
        return self.summary(self.samples, self.max_mhz, self.source, self.bus)

    @staticmethod
    def summary(samples, max_mhz, source, bus):
        if not samples:
            return None
        sm = [x for x, _ in samples]
        reasons = sorted({n for _, names in samples for n in names})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max_mhz, "reasons": reasons,
                "samples": len(sm), "sm_mhz_min": min(sm), "source": source, "gpu_pci": bus}


# ---------------------------------------------------------------- our arm --

def run_ours(args, rank, world):
    from fp8_mxfp4_grouped_gb300 import hg
    from synth import make_case
    from synth.inputs import CONFIGS

    dev = torch.device("cuda")
    cfg = CONFIGS[args.config]
    Ms = args.Ms or cfg["Ms"]
    peaks = load_peaks()
    fp8_peak = peaks["bf16"] * FP8_OVER_BF16
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(l2, dev)
    stream = torch.cuda.Stream()

    cases = []
    for M in Ms:
        c = make_case(args.config, M, projection=args.proj, routing=args.routing, device=dev)
        R = c.R
        bufs = device_buffers(c, dev, hg)
        e_act = active_experts(bufs, c, stream, hg)
        # pinned host copies for the end-to-end leg
        host = dict(ids=torch.from_numpy(c.topk_ids).pin_memory(),
                    a=c.a_fp8.cpu().pin_memory(), a_s=c.a_scale.cpu().pin_memory(),
                    out=torch.empty((R, c.N), dtype=torch.bfloat16).pin_memory())
        flops, byts = algorithmic(R, e_act, c.E, c.N, c.K)
        cases.append(dict(M=M, c=c, R=R, e_act=e_act, flops=flops, bytes=byts, bufs=bufs,
                          host=host))

    def launch(cs, s):
        b = cs["bufs"]
        c = cs["c"]
        hg.hg_plan_expert_offsets(b["ids"], c.E, b["off"], b["s2d"], b["d2s"], b["ws"], stream=s)
        hg.hg_grouped_w4a8_gemm(c.a_fp8, c.a_scale, c.w_fp4, c.w_scale, b["off"], out=b["out"],
                                stream=s)

    # One step: for every M, an L2 flush, then the routing plan and the GEMM
    # in one event bracket.  The GEMM is launched with programmatic dependent
    # launch, so its prologue overlaps the plan's last kernel; an event
    # between the two would serialise them again.  The split into plan and
    # GEMM time comes from a separate, untimed pass (time_breakdown).
    def one_step(record):
        times = []
        for cs in cases:
            with torch.cuda.stream(stream):
                flush(cs["M"])
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                launch(cs, stream)
                e1.record(stream)
            times.append((e0, e1))
        if record is not None:
            record.append(times)

    for _ in range(args.warmup):
        one_step(None)
    torch.cuda.synchronize()
    st, detail = hg.hg_get_device_status()
    if st != hg.HG_OK:
        raise RuntimeError(f"device status {st} detail {detail} after warm-up")

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    time.sleep(0.3)
    recs = []
    barrier(world)
    torch.cuda.synchronize()
    gc.disable()   # no collector pause inside the timed region
    t_wall0 = time.perf_counter()
    torch.cuda.nvtx.range_push("timed")      # lets a profiler select exactly these launches
    for _ in range(args.steps):
        one_step(recs)
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize()
    barrier(world)
    t_wall = time.perf_counter() - t_wall0
    gc.enable()
    clk = clocks.stop()

    step_us = [[] for _ in cases]
    for times in recs:
        for i, (e0, e1) in enumerate(times):
            step_us[i].append(e0.elapsed_time(e1) * 1e3)
    st, detail = hg.hg_get_device_status()
    if st != hg.HG_OK:
        raise RuntimeError(f"device status {st} detail {detail} after timing")

    device_s = sum(sum(t) for t in step_us) * 1e-6   # all K steps
    flops_step = sum(cs["flops"] for cs in cases)
    dev_max = reduce_scalar(device_s, "max", world)
    flops_all = reduce_scalar(flops_step * args.steps, "sum", world)
    value = flops_all / dev_max / 1e12

    # Breakdown (outside the timed region): plan alone, plan + GEMM, GEMM alone.
    reps = max(5, min(args.steps, 20))
    sweep = []
    for cs in cases:
        p, pg, ga = time_breakdown(flush, stream, hg, cs["c"], cs["bufs"], reps)
        e = sweep_entry(cs, pg, p, ga, peaks, fp8_peak)
        e["plan_gemm_us_timed"] = round(statistics.median(step_us[len(sweep)]), 2)
        sweep.append(e)
    # The roofline object is the GEMM kernel timed alone in its own bracket.
    dom = max(range(len(cases)), key=lambda i: sweep[i]["gemm_alone_us"])
    dcs = cases[dom]
    dg = sweep[dom]["gemm_alone_us"] * 1e-6
    if sweep[dom]["bound"] == "tensor":
        roof = dict(bound="tensor", achieved=round(dcs["flops"] / dg / 1e12, 1),
                    peak=round(fp8_peak, 1), unit="TFLOP/s")
    else:
        roof = dict(bound="hbm", achieved=round(dcs["bytes"] / dg / 1e9, 1),
                    peak=peaks["hbm_gbs"], unit="GB/s")
    roof["frac"] = round(roof["achieved"] / roof["peak"], 3)
    roof["traffic"] = measured_traffic(dcs["M"]) if default_workload(args) else None
    roof["launch"] = (f"GEMM at M={dcs['M']} (largest share of the step), timed alone in "
                      f"its own event bracket")
    roof["peak_source"] = (f"{peaks['source']}: bf16 {peaks['bf16']} TFLOP/s x{FP8_OVER_BF16} "
                           f"nominal fp8/bf16" if roof["bound"] == "tensor"
                           else f"{peaks['source']} HBM copy")
    roof["sweep_roof_time_frac"] = round(
        sum(max(cs["bytes"] / (peaks["hbm_gbs"] * 1e9), cs["flops"] / (fp8_peak * 1e12))
            for cs in cases) / (sum(e["gemm_alone_us"] for e in sweep) * 1e-6), 3)

    # ---- end to end: every batch through hg_grouped_w4a8_gemm_host, which
    # takes the ids, activations, scales and output in pinned host memory and
    # makes the copies itself (ids, A and scales up, plan, GEMM, output down,
    # all on one stream).  The sweep's batches are independent: they go to
    # three streams in turn, so one batch's uploads overlap another's GEMM
    # and a third's download.
    e2e = None
    if not args.no_e2e:
        e_streams = [torch.cuda.Stream() for _ in range(max(1, args.e2e_streams))]
        for cs in cases:
            c = cs["c"]
            cs["host_ws"] = torch.empty(
                hg.hg_gemm_host_workspace_bytes(c.M, c.top_k, c.E, c.N, c.K), dtype=torch.uint8,
                device=dev)

        def e2e_events():
            return (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                    [torch.cuda.Event() for _ in e_streams])

        def e2e_step(events):
            e0, e1, ends = events
            e0.record(stream)
            for s in e_streams:
                s.wait_event(e0)
            for i, cs in enumerate(cases):
                c, h = cs["c"], cs["host"]
                hg.hg_grouped_w4a8_gemm_host(h["ids"], h["a"], h["a_s"], c.w_fp4, c.w_scale,
                                             c.E, h["out"], cs["host_ws"],
                                             stream=e_streams[i % len(e_streams)])
            for s, ev in zip(e_streams, ends):
                ev.record(s)
                stream.wait_event(ev)
            e1.record(stream)
            return e0, e1

        for _ in range(max(3, args.warmup)):
            e2e_step(e2e_events())
        torch.cuda.synchronize()
        e2e_steps = min(args.steps, 20)
        events = [e2e_events() for _ in range(e2e_steps)]
        step_s = []
        gc.disable()   # no collector pause inside the timed steps
        for k in range(e2e_steps):
            e0, e1 = e2e_step(events[k])
            torch.cuda.synchronize()
            step_s.append(e0.elapsed_time(e1) * 1e-3)
        gc.enable()
        # The step is a median over the timed steps.  In repeated runs of
        # this loop about one step in 20-60 took 10-30 ms instead of 3 (with
        # one stream or three, in either batch order; the other steps varied
        # by under 1 %), so a plain mean over 20 steps swung by a third
        # between runs.  The mean is reported beside it.
        med = statistics.median(step_s)
        tot = reduce_scalar(med * e2e_steps, "max", world)
        tot_mean = reduce_scalar(sum(step_s), "max", world)
        flops_e2e = reduce_scalar(flops_step * e2e_steps, "sum", world)
        bi = sum(cs["c"].topk_ids.nbytes + cs["c"].a_fp8.numel() + cs["c"].a_scale.numel()
                 for cs in cases)
        bo = sum(cs["host"]["out"].numel() * 2 for cs in cases)
        link = host_link_gbs(cases[-1], dev)
        e2e = dict(value=round(flops_e2e / tot / 1e12, 2), unit=UNIT, h2d_bytes_per_step=int(bi),
                   d2h_bytes_per_step=int(bo), ms_per_step=round(tot / e2e_steps * 1e3, 3),
                   step_statistic="median of the timed steps",
                   value_mean=round(flops_e2e / tot_mean / 1e12, 2),
                   ms_per_step_mean=round(tot_mean / e2e_steps * 1e3, 3),
                   steps_over_2x_median=sum(t > 2 * med for t in step_s),
                   host_link_gbs=link,
                   copy_floor_ms=round((bi + bo) / (link["both"] * 1e9) * 1e3, 3),
                   note="hg_grouped_w4a8_gemm_host per batch (pinned host buffers, the library "
                        f"copies); batches on {len(e_streams)} streams in turn")

    moe_io = None if args.no_moe_io else time_moe_io(cases[-1], flush, stream, peaks, hg)

    others = None
    clk_others = None
    if default_workload(args) and not args.no_other_workloads:
        # clocks sampled while the other workloads run, for reading their numbers
        sampler = ClockSampler(torch.cuda.current_device())
        sampler.start()
        others = time_other_workloads(flush, stream, peaks, fp8_peak, hg,
                                      reps=max(5, min(args.steps, 20)))
        clk_others = sampler.stop()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args)


    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dev_max / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8e4m3 x fp4e2m1 -> f32 acc -> bf16",
        "data": "synthetic (seeded routing, N(0,1) values quantised as the configs state)",
        "config": line_config(args, world),
        "sweep": sweep,
        "other_workloads": others,
        "targets": target_summary(sweep, others or []),
        "roofline": roof,
        "moe_io": moe_io,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": sum(hg.hg_plan_launches(cs["M"], cs["c"].top_k, cs["c"].E) + 1
                            for cs in cases) * args.steps,
        "clocks": clk,
        "clocks_other_workloads": clk_others,
        "wall_s_timed": round(t_wall, 3),
    }
    return line


def time_moe_io(cs, flush, stream, peaks, hg, reps=20):
    """Device time of the kernels around the GEMM at the sweep's largest M:
    BF16 -> E4M3 quantise + gather into sorted order, and the top-k combine.
    Both are HBM-bound; roofline = algorithmic bytes / HBM peak."""
    c, b = cs["c"], cs["bufs"]
    M, K, N, k, R = c.M, c.K, c.N, c.top_k, cs["R"]
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    x = torch.randn((M, K), generator=gen, device="cuda").to(torch.bfloat16)
    w = torch.rand((M, k), generator=gen, device="cuda")
    a = torch.empty((R, K), dtype=torch.uint8, device="cuda")
    s = torch.empty((R, K // 128), dtype=torch.uint8, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    hg.hg_plan_expert_offsets(b["ids"], c.E, b["off"], b["s2d"], b["d2s"], b["ws"], stream=stream)

    def timed(fn):
        ts = []
        for it in range(reps + 3):
            with torch.cuda.stream(stream):
                flush(it)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
            if it >= 3:
                ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.median(x0.elapsed_time(x1) for x0, x1 in ts) * 1e3

    tq = timed(lambda: hg.hg_quantize_gather_acts(x, k, b["s2d"], a, s, stream=stream))
    tqs = timed(lambda: hg.hg_quantize_scatter_acts(x, k, b["d2s"], a, s, stream=stream))
    tc = timed(lambda: hg.hg_combine_topk(b["out"], b["d2s"], w, out, stream=stream))
    bq = M * K * 2 + R * 4 + R * K + R * K / 128     # tokens read once, codes written once per row
    bc = R * N * 2 + R * 4 + M * k * 4 + M * N * 2
    hbm = peaks["hbm_gbs"]
    return {"M": M, "quantize_scatter_us": round(tqs, 2),
            "quantize_scatter_gbs": round(bq / tqs / 1e3, 1),
            "quantize_scatter_roof_frac": round(bq / tqs / 1e3 / hbm, 3),
            "quantize_gather_us": round(tq, 2), "quantize_gather_gbs": round(bq / tq / 1e3, 1),
            "quantize_gather_roof_frac": round(bq / tq / 1e3 / hbm, 3),
            "combine_us": round(tc, 2), "combine_gbs": round(bc / tc / 1e3, 1),
            "combine_roof_frac": round(bc / tc / 1e3 / hbm, 3),
            "bytes": {"quantize": int(bq), "combine": int(bc)}}


# ------------------------------------------------------------ oracle arms --

def default_workload(args):
    """The workload the headline line is quoted on (configuration 1, gate/up, skewed routing)."""
    return args.config == CONFIG_ID and args.proj in (None, "gate_up") and \
        args.routing in (None, "biased")


def line_config(args, world):
    """The `config` object both arms print: the workload, its shapes and the L2 rule."""
    from synth.inputs import CONFIGS
    cfg = CONFIGS[args.config]
    Ms = args.Ms or cfg["Ms"]
    proj = args.proj or list(cfg["proj"])[0]
    routing = args.routing or cfg["routing"][0]
    N, K = cfg["proj"][proj]
    if default_workload(args):
        workload, routing_desc = WORKLOAD, "biased (unbalanced)"
    else:
        workload = (f"{cfg['name']} {proj} E={cfg['E']} top{cfg['top_k']} N={N} K={K} "
                    f"{routing}, M sweep {Ms[0]}..{Ms[-1]}")
        routing_desc = routing
    return {"workload": workload, "E": cfg["E"], "top_k": cfg["top_k"], "N": N, "K": K,
            "Ms": Ms, "routing": routing_desc, "l2": L2Flush.DESCRIPTION,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


class OracleSample:
    """The CPU oracle as it stands, on a bounded sample of the workload: the
    routing plan and the full float64 GEMM (every expert) of the sweep's
    smallest M.  Both the cpu_baseline leg and the --impl reference arm time
    exactly this."""

    def __init__(self, args):
        from synth import make_case
        from synth.inputs import CONFIGS
        M = (args.Ms or CONFIGS[args.config]["Ms"])[0]
        c = make_case(args.config, M, projection=args.proj, routing=args.routing, device="cpu",
                      cache_weights=False)
        self.c = c
        self.a, self.a_s = c.a_fp8.numpy(), c.a_scale.numpy()
        self.w, self.w_s = c.w_fp4.numpy(), c.w_scale.numpy()
        self.flops = 2.0 * c.R * c.N * c.K
        self.desc = (f"{c.projection} M={M} (R={c.R}): oracle plan + full float64 GEMM over all "
                     f"{c.E} experts per step; numpy decode single-threaded, matmul on the host "
                     f"BLAS threads ({os.cpu_count()} cores)")

    def step(self):
        from oracle import gemm as G
        from oracle.plan import plan_expert_offsets
        c = self.c
        off, *_ = plan_expert_offsets(c.topk_ids, c.E)
        G.grouped_w4a8_gemm(self.a, self.a_s, self.w, self.w_s, off, c.E, c.N, c.K)


def cpu_baseline(args):
    """The oracle sample timed on the host cores: the median of 3 reps when one
    rep takes under 10 s, else that one rep."""
    smp = OracleSample(args)
    ts = []
    while len(ts) < 3:
        t0 = time.perf_counter()
        smp.step()
        ts.append(time.perf_counter() - t0)
        if ts[0] >= 10.0:
            break
    dt = statistics.median(ts)
    return {"value": round(smp.flops / dt / 1e12, 6), "unit": UNIT, "cores": os.cpu_count(),
            "kind": "oracle", "reps": len(ts), "s_per_rep": round(dt, 2),
            "sample": smp.desc}


def run_reference(args, rank, world):
    """--impl reference: the oracle sample timed on the host cores (rank 0 only),
    W untimed steps then K timed ones."""
    if rank != 0:
        return None
    smp = OracleSample(args)
    for _ in range(args.warmup):
        smp.step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        smp.step()
    dt = time.perf_counter() - t0
    v = smp.flops * args.steps / dt / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 6), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded routing, N(0,1) values quantised as the configs state)",
        "config": line_config(args, world),
        "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "kind": "oracle",
                         "cores": os.cpu_count(), "sample": smp.desc},
        "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--Ms", type=lambda s: [int(x) for x in s.split(",")], default=None)
    # another configuration's shapes (for profiling; the headline is configuration 1)
    ap.add_argument("--config", type=int, default=CONFIG_ID)
    ap.add_argument("--proj", default=None)
    ap.add_argument("--routing", default=None)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-streams", type=int, default=3,
                    help="streams the end-to-end leg deals its batches to, in turn")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-moe-io", action="store_true")
    ap.add_argument("--no-other-workloads", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    rank, world, _ = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
