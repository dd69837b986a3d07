"""bench.py's per-shape bookkeeping on CPU: algorithmic bytes and FLOPs, the
roofline fractions of one sweep entry (GEMM in the plan -> GEMM sequence and
alone), and the two target summaries."""
import pytest

import bench

PEAKS = {"hbm_gbs": 8000.0}
FP8 = 4000.0   # TFLOP/s


def test_algorithmic_counts_each_operand_once():
    R, E_act, E, N, K = 512, 10, 32, 4096, 6144
    flops, byts = bench.algorithmic(R, E_act, E, N, K)
    assert flops == 2 * R * N * K
    weights = E_act * N * K // 2 + E_act * N * K // 32      # E2M1 codes + E8M0 scales
    acts = R * K + R * K // 128                              # E4M3 codes + E8M0 scales
    assert byts == weights + acts + 2 * R * N + 4 * (E + 1)  # BF16 out, offsets


def test_sweep_entry_fractions():
    flops, byts = 2.0e12 * 1e-3, 4.0e9 * 1e-3     # 2 GFLOP, 4 MB
    cs = dict(M=64, R=512, e_act=7, flops=flops, bytes=byts)
    # t_hbm = 4e6 / 8e12 = 0.5 us; t_fp8 = 2e9 / 4e15 = 0.5 us
    e = bench.sweep_entry(cs, pg_us=3.0, p_us=1.0, ga_us=4.0, peaks=PEAKS, fp8_peak=FP8)
    assert e["gemm_us"] == pytest.approx(2.0) and e["gemm_alone_us"] == 4.0
    assert e["plan_gemm_us"] == 3.0 and e["plan_us"] == 1.0
    assert e["roof_frac"] == pytest.approx(0.25) and e["roof_frac_alone"] == pytest.approx(0.125)
    assert e["hbm_frac"] == pytest.approx(0.25) and e["hbm_frac_alone"] == pytest.approx(0.125)
    assert e["tflops"] == pytest.approx(1000.0)
    # tensor-bound when the FLOP time is longer
    cs2 = dict(cs, flops=4 * flops)
    e2 = bench.sweep_entry(cs2, 3.0, 1.0, 4.0, PEAKS, FP8)
    assert e2["bound"] == "tensor" and e2["roof_frac"] == pytest.approx(1.0)
    assert e2["hbm_frac"] == pytest.approx(0.25)


def _row(M, roof, hbm, roof_a, hbm_a):
    return dict(M=M, roof_frac=roof, hbm_frac=hbm, roof_frac_alone=roof_a, hbm_frac_alone=hbm_a)


def test_target_summary_uses_the_sequence_and_reports_alone():
    head = [_row(64, 0.8, 0.8, 0.7, 0.7), _row(2048, 0.9, 0.3, 0.85, 0.28)]
    others = [{"config": 3, "projection": "w2", "routing": "uniform",
               "sweep": [_row(8, 0.56, 0.56, 0.45, 0.45), _row(256, 0.49, 0.49, 0.41, 0.41)]},
              {"config": 4, "projection": "down", "routing": "biased",
               "sweep": [_row(4096, 0.78, 0.36, 0.77, 0.36)]}]
    t = bench.target_summary(head, others)
    small, big = t["m_le_256_min_hbm_frac"], t["m_ge_4096_min_roof_frac"]
    assert small["value"] == 0.49 and small["at"] == "config3 w2 uniform M=256"
    assert small["below"] == ["config3 w2 uniform M=256: 0.49"]
    assert small["gemm_alone"]["value"] == 0.41 and small["gemm_alone"]["below"] == 2
    assert big["value"] == 0.78 and big["below"] == [] and big["gemm_alone"]["below"] == 0
    assert big["target"] == 0.70 and small["target"] == 0.50
