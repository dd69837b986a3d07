"""The seeded generator: determinism, routing properties, and the
quantisation rules stated for the workloads (scale 2^ceil(log2(amax/qmax)),
round-to-nearest-even onto the element grid)."""
import numpy as np
import torch

from oracle.formats import decode_e2m1_packed, decode_e4m3, decode_e8m0
from synth import make_case, make_routing, quantize_acts, quantize_weights
from synth.inputs import CONFIGS


def test_routing_deterministic_and_distinct():
    for mode in ("uniform", "biased"):
        a = make_routing(300, 32, 8, mode, seed=5)
        b = make_routing(300, 32, 8, mode, seed=5)
        assert np.array_equal(a, b)
        assert a.dtype == np.int32 and a.shape == (300, 8)
        assert all(len(set(row)) == 8 for row in a.tolist())
        assert a.min() >= 0 and a.max() < 32


def test_biased_routing_is_skewed_uniform_is_not():
    ub = np.bincount(make_routing(4096, 32, 8, "biased", 1).ravel(), minlength=32)
    un = np.bincount(make_routing(4096, 32, 8, "uniform", 1).ravel(), minlength=32)
    assert ub.max() / ub.mean() > 2.0
    assert un.max() / un.mean() < 1.2


def test_act_quantiser_rule():
    g = torch.Generator().manual_seed(3)
    x = torch.randn(64, 512, generator=g) * torch.exp2(torch.randint(-8, 8, (64, 1), generator=g).float())
    x[3, :128] = 0.0                                   # an all-zero group
    codes, sc = quantize_acts(x)
    assert codes.dtype == torch.uint8 and sc.shape == (64, 4)
    assert not np.any((codes.numpy() & 0x7F) == 0x7F)   # no NaN codes
    amax = x.reshape(64, 4, 128).abs().amax(-1).double().numpy()
    s = decode_e8m0(sc.numpy())
    nz = amax > 0
    assert np.all(amax[nz] <= 448 * s[nz]) and np.all(amax[nz] > 224 * s[nz])
    assert sc[3, 0] == 127
    deq = decode_e4m3(codes.numpy()) * np.repeat(s, 128, axis=1)
    err = np.abs(deq - x.double().numpy())
    # RNE onto E4M3: error at most half a quantum, quantum = 2^(floor(log2|q|)-3), >= 2^-9
    q = np.abs(x.double().numpy()) / np.repeat(s, 128, axis=1)
    quantum = np.maximum(2.0 ** (np.floor(np.log2(np.maximum(q, 1e-300))) - 3), 2.0 ** -9)
    assert np.all(err <= 0.5 * quantum * np.repeat(s, 128, axis=1) * (1 + 1e-12))


def test_weight_quantiser_rule_and_ties():
    q = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.75, 6.0, -6.0, 0.3, 2.4] + [0.0] * 20)
    packed, sc = quantize_weights(q.reshape(1, 32) * 1.0)
    assert sc.item() == 127                 # amax 6 -> scale 1
    vals = decode_e2m1_packed(packed.numpy())[0, :12]
    assert vals.tolist() == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, -1.0, 6.0, -6.0, 0.5, 2.0]


def test_weight_quantiser_scale():
    g = torch.Generator().manual_seed(4)
    w = torch.randn(2, 128, 256, generator=g)
    packed, sc = quantize_weights(w)
    assert packed.shape == (2, 128, 128) and sc.shape == (2, 128, 8)
    amax = w.reshape(2, 128, 8, 32).abs().amax(-1).double().numpy()
    s = decode_e8m0(sc.numpy())
    assert np.all(amax <= 6 * s) and np.all(amax > 3 * s)


def test_case_shapes():
    c = make_case(0, 16)
    assert (c.E, c.top_k, c.N, c.K, c.R) == (4, 2, 256, 512, 32)
    assert c.a_fp8.shape == (32, 512) and c.a_scale.shape == (32, 4)
    assert c.w_fp4.shape == (4, 256, 256) and c.w_scale.shape == (4, 256, 16)
    c2 = make_case(0, 16)
    assert torch.equal(c.a_fp8, c2.a_fp8) and np.array_equal(c.topk_ids, c2.topk_ids)
    assert set(CONFIGS) == {0, 1, 2, 3, 4}
