"""Seeded synthetic workloads with the shapes of the pages' benchmarks.

Shapes follow humming PR #129 ("perf(sm90): size grouped W4A8 tiles per
expert", result tables: gate/up N=4096 K=6144 and down N=6144 K=2048, E=32,
top-8, default unbalanced routing) and humming PR #58 ("Tune SM90 small-M FP4
schedules", H200 performance table: E=12, top-8, balanced routing, W13
N=6144 K=3584 and W2 N=3584 K=3072).

Recipe (identical on every machine for the routing; values come from a
seeded torch generator on the device that draws them):

* routing, "uniform": per token, k distinct experts uniformly at random
  (argsort of i.i.d. uniform keys);  "biased": per-token logits N(0,1) plus a
  per-expert bias N(0,1) drawn once (seed 12345), top-k distinct by logit.
  numpy PCG64, seed 1000*config + M.
* activations: N(0,1) float32 [R, K] (R = M*k routed rows, generated directly
  in sorted order since rows are i.i.d.), quantised per row per 128-K group:
  scale 2^ceil(log2(amax/448)), codes = E4M3 round-to-nearest-even of x/scale.
* weights: N(0,1) float32 [E, N, K], quantised per output column per 32-K
  group: scale 2^ceil(log2(amax/6)), codes = E2M1 round-to-nearest-even of
  x/scale (ties to the even code), two codes per byte, element 2j in the low
  nibble.  An all-zero group gets scale code 127.

Nothing here decodes codes back to values or multiplies operands.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

#: The five workload configurations (shapes, expert counts, routing).
CONFIGS = {
    0: dict(name="tiny", E=4, top_k=2, proj={"tiny": (256, 512)}, Ms=[16],
            routing=["uniform"]),
    1: dict(name="gate_up", E=32, top_k=8, proj={"gate_up": (4096, 6144)},
            Ms=[64, 256, 512, 768, 1152, 1536, 2048], routing=["biased"]),
    2: dict(name="down", E=32, top_k=8, proj={"down": (6144, 2048)},
            Ms=[64, 256, 512, 1024, 1536, 4096, 16384], routing=["biased"]),
    3: dict(name="small_m_few_experts", E=12, top_k=8,
            proj={"w13": (6144, 3584), "w2": (3584, 3072)},
            Ms=[1, 4, 8, 64, 256], routing=["uniform"]),
    4: dict(name="large_m", E=32, top_k=8,
            proj={"gate_up": (4096, 6144), "down": (6144, 2048)},
            Ms=[4096, 16384], routing=["uniform", "biased"]),
}

BIAS_SEED = 12345
A_GROUP = 128
W_GROUP = 32
E4M3_MAX = 448.0
E2M1_MAX = 6.0


def make_routing(M: int, E: int, top_k: int, mode: str, seed: int) -> np.ndarray:
    """int32 [M, top_k] expert ids, k distinct per token."""
    if top_k > E:
        raise ValueError("top_k > E")
    rng = np.random.Generator(np.random.PCG64(seed))
    if mode == "uniform":
        keys = rng.random((M, E))
        ids = np.argsort(keys, axis=1, kind="stable")[:, :top_k]
    elif mode == "biased":
        bias = np.random.Generator(np.random.PCG64(BIAS_SEED)).standard_normal(E)
        logits = rng.standard_normal((M, E)) + bias[None, :]
        ids = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    else:
        raise ValueError(f"unknown routing mode {mode!r}")
    return np.ascontiguousarray(ids.astype(np.int32))


def _pow2_exponent(amax: torch.Tensor, qmax: float) -> torch.Tensor:
    """Smallest integer e with amax <= qmax*2^e (0 for amax == 0), in [-127, 127]."""
    a = amax.to(torch.float64)
    safe = torch.where(a > 0, a, torch.ones_like(a))
    e = torch.ceil(torch.log2(safe / qmax))
    # log2 may be off by one ulp near powers of two: settle the inequality exactly
    e = torch.where(safe > qmax * torch.exp2(e), e + 1, e)
    e = torch.where(safe <= qmax * torch.exp2(e - 1), e - 1, e)
    e = torch.where(a > 0, e, torch.zeros_like(e))
    return e.clamp(-127, 127).to(torch.int32)


def quantize_acts(x: torch.Tensor):
    """float32 [R, K] -> (E4M3 codes uint8 [R, K], E8M0 codes uint8 [R, K/128])."""
    R, K = x.shape
    g = x.reshape(R, K // A_GROUP, A_GROUP)
    e = _pow2_exponent(g.abs().amax(dim=-1), E4M3_MAX)
    q = g / torch.exp2(e.to(torch.float32)).unsqueeze(-1)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8).reshape(R, K)
    return codes.contiguous(), (e + 127).to(torch.uint8).contiguous()


# E2M1 magnitudes by code 0..7 and the midpoints between neighbours.
_E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def _e2m1_codes(q: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even onto the E2M1 grid; |q| <= 6 assumed. uint8 codes."""
    mag = q.abs()
    code = torch.zeros(q.shape, dtype=torch.uint8, device=q.device)
    for i, mid in enumerate(_E2M1_MIDPOINTS):
        # a tie between codes i and i+1 goes to the even one
        up = (mag > mid) | ((mag == mid) & (i % 2 == 1))
        code += up.to(torch.uint8)
    sign = (q < 0).to(torch.uint8) << 3
    return code | sign


def quantize_weights(w: torch.Tensor):
    """float32 [..., N, K] -> (packed E2M1 uint8 [..., N, K/2], E8M0 uint8 [..., N, K/32])."""
    *lead, N, K = w.shape
    g = w.reshape(*lead, N, K // W_GROUP, W_GROUP)
    e = _pow2_exponent(g.abs().amax(dim=-1), E2M1_MAX)
    q = g / torch.exp2(e.to(torch.float32)).unsqueeze(-1)
    codes = _e2m1_codes(q).reshape(*lead, N, K)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    return packed.contiguous(), (e + 127).to(torch.uint8).contiguous()


def _generator(device, seed: int) -> torch.Generator:
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return gen


def make_acts(R: int, K: int, seed: int, device="cpu", chunk_rows: int = 16384):
    """Quantised N(0,1) activations: (a_fp8 [R, K], a_scale [R, K/128])."""
    gen = _generator(device, seed)
    a = torch.empty((R, K), dtype=torch.uint8, device=device)
    s = torch.empty((R, K // A_GROUP), dtype=torch.uint8, device=device)
    for r0 in range(0, R, chunk_rows):
        r1 = min(R, r0 + chunk_rows)
        x = torch.randn((r1 - r0, K), generator=gen, device=device, dtype=torch.float32)
        a[r0:r1], s[r0:r1] = quantize_acts(x)
    return a, s


def make_weights(E: int, N: int, K: int, seed: int, device="cpu"):
    """Quantised N(0,1) weights: (w_fp4 [E, N, K/2], w_scale [E, N, K/32])."""
    gen = _generator(device, seed)
    w = torch.empty((E, N, K // 2), dtype=torch.uint8, device=device)
    s = torch.empty((E, N, K // W_GROUP), dtype=torch.uint8, device=device)
    for e in range(E):
        x = torch.randn((N, K), generator=gen, device=device, dtype=torch.float32)
        w[e], s[e] = quantize_weights(x)
    return w, s


@dataclass
class Case:
    config_id: int
    M: int
    E: int
    top_k: int
    N: int
    K: int
    routing: str
    projection: str
    topk_ids: np.ndarray            # int32 [M, top_k]
    a_fp8: torch.Tensor             # uint8 [R, K]
    a_scale: torch.Tensor           # uint8 [R, K/128]
    w_fp4: torch.Tensor             # uint8 [E, N, K/2]
    w_scale: torch.Tensor           # uint8 [E, N, K/32]
    meta: dict = field(default_factory=dict)

    @property
    def R(self) -> int:
        return self.M * self.top_k


def case_seed(config_id: int, M: int) -> int:
    return 1000 * config_id + M


def weight_seed(config_id: int, proj_index: int) -> int:
    return 7 + 100 * config_id + proj_index


_WEIGHT_CACHE: dict = {}


def make_case(config_id: int, M: int, projection: str | None = None,
              routing: str | None = None, device="cpu", cache_weights=True) -> Case:
    """Build one seeded workload of a configuration."""
    cfg = CONFIGS[config_id]
    projs = list(cfg["proj"].keys())
    projection = projection or projs[0]
    routing = routing or cfg["routing"][0]
    N, K = cfg["proj"][projection]
    E, k = cfg["E"], cfg["top_k"]
    seed = case_seed(config_id, M)
    ids = make_routing(M, E, k, routing, seed)
    a, a_s = make_acts(M * k, K, seed + 1, device=device)
    key = (config_id, projection, str(device))
    if cache_weights and key in _WEIGHT_CACHE:
        w, w_s = _WEIGHT_CACHE[key]
    else:
        w, w_s = make_weights(E, N, K, weight_seed(config_id, projs.index(projection)),
                              device=device)
        if cache_weights:
            _WEIGHT_CACHE.clear()
            _WEIGHT_CACHE[key] = (w, w_s)
    return Case(config_id, M, E, k, N, K, routing, projection, ids, a, a_s, w, w_s)


def clear_cache():
    _WEIGHT_CACHE.clear()
