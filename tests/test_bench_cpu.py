"""Host logic of bench.py that needs no GPU: the routing report against the
oracle's near-ties, the clock summary and the choice of the FFN's roofline."""
import numpy as np
import pytest

import bench
from synth import workloads


def test_routing_report_counts_near_ties_and_mismatches():
    ids = np.array([[0, 1], [2, 3], [4, 5], [6, 7]], dtype=np.int32)
    ref = {"ids": ids.copy(), "margin": np.array([1e-6, 0.5, 2e-5, 0.3])}
    gpu = ids.copy()
    gpu[0] = [1, 0]            # differs at a near-tie
    gpu[1] = [2, 4]            # differs away from one
    r = bench.routing_report(gpu, ref)
    assert r["tokens"] == 4 and r["near_tie_tokens"] == 2
    assert r["mismatched_tokens"] == 2 and r["mismatched_away_from_near_tie"] == 1


def test_clock_summary_uses_loaded_samples_and_reasons():
    c = bench.ClockSampler(0)
    c.kind = "test"
    c.thread = None   # samples as nvidia-smi takes them: filtered by power
    c.rows = [(1000.0, 2032.0, 150.0, 0x0), (2032.0, 2032.0, 900.0, 0x0), (1980.0, 2032.0, 1100.0, 0x4),
              (2032.0, 2032.0, 950.0, 0x0)]
    s = c.summary()
    assert s["sm_mhz"] == 2032.0 and s["samples_under_load"] == 3
    assert s["reasons"] == ["sw_power_cap"] and s["sm_max_mhz"] == 2032.0


@pytest.mark.parametrize("name,bound", [("mixtral_8x7b", "tensor"), ("deepseek_v3", "hbm"),
                                        ("deepseek_v3_decode_T32", "hbm")])
def test_ffn_roofline_bound_follows_arithmetic_intensity(name, bound):
    w = workloads.ALL[name]
    rows = w.T * w.K
    touched = min(w.E, rows)
    work = {"ffn_bytes": touched * 3 * w.h * w.I * 2 + rows * (2 * w.h + 2 * w.I) * 2,
            "ffn_flops": 6.0 * w.h * w.I * rows}
    peaks = {"hbm_gbs": 6500.0, "bf16_tflops_sustained": 1380.0}
    r = bench.ffn_roofline(w, work, 2.0, peaks, "measured")
    assert r["bound"] == bound
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
