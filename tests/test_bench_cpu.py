"""Host-side measurement logic of bench.py, on CPU: the algorithmic FLOP
counts the throughput is quoted in, and the parsing of the clock samples that
decide whether a timed run is kept."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import synth  # noqa: E402


def _counted_flops(wl):
    """Multiply-adds counted product by product from an explicit selection:
    every query row meets every token of each of its K selected cubes."""
    rng = np.random.default_rng(0)
    per_head_pairs = 0
    for _ in range(wl.BH):
        lists = [rng.choice(wl.Nc, size=wl.topk, replace=False) for _ in range(wl.Nc)]
        per_head_pairs += sum(64 * 64 * len(lst) for lst in lists)     # (query row, key row) pairs
    pairs = per_head_pairs
    fwd = 2 * pairs * wl.d * 2            # S = Q K^T and O = P V: d MACs each per pair
    bwd = 2 * pairs * wl.d * 5            # S (recomputed), dP, dV, dQ, dK
    coarse = 2 * wl.BH * wl.Nc * wl.Nc * wl.d * 7   # S_c, O_c; S_c again, dP_c, dQ_c, dK_c, dV_c
    return fwd, bwd, coarse


@pytest.mark.parametrize("name", ["tiny", "small", "wan1.3b"])
def test_step_flops_match_a_product_by_product_count(name):
    wl = synth.WORKLOADS[name]
    fwd, bwd, coarse = _counted_flops(wl)
    got = bench.step_flops(wl)
    assert got["fine_fwd"] == pytest.approx(fwd, rel=1e-12)
    assert got["fine_bwd"] == pytest.approx(bwd, rel=1e-12)
    assert got["coarse"] == pytest.approx(coarse, rel=1e-12)
    assert got["total"] == pytest.approx(fwd + bwd + coarse, rel=1e-12)


def test_bench_layer_fine_forward_flops():
    """The figure the roofline quotes for the 32K-token layer: 12 heads x 32768
    queries x 154 cubes x 64 keys x 128 channels x 4 FLOP."""
    assert bench.step_flops(synth.WORKLOADS["wan1.3b"])["fine_fwd"] == 1984274890752.0


def _sampler(lines):
    s = bench.ClockSampler(0)
    s.lines = list(lines)
    return s


def test_clock_summary_median_and_no_reasons():
    s = _sampler(["2070, 2070, 900.1, Not Active, Not Active, Not Active, Not Active",
                  "2055, 2070, 950.0, Not Active, Not Active, Not Active, Not Active",
                  "2070, 2070, 980.2, Not Active, Not Active, Not Active, Not Active"])
    got = s.summary()
    assert got == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3}


def test_clock_summary_reports_each_active_reason():
    s = _sampler(["1800, 2070, 1400.0, Not Active, Not Active, Not Active, Active",
                  "1700, 2070, 1400.0, Active, Not Active, Active, Not Active",
                  "garbage line",
                  "[N/A], 2070, 1400.0, Not Active, Not Active, Not Active, Not Active"])
    got = s.summary()
    assert got["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert got["samples"] == 2 and got["sm_mhz"] == 1750.0


def test_clock_summary_without_samples():
    assert _sampler([]).summary()["reasons"] == ["no samples"]


def test_peaks_read_both_measurements():
    p = bench.load_peaks()
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        assert p["source"] == "fallback" and p["burst"] > p["sustained"]
        return
    import json
    with open(path) as f:
        m = json.load(f)
    assert p["burst"] == m["bf16_tflops"]
    assert p["sustained"] == (m.get("bf16_tflops_sustained") or m["bf16_tflops"])
    assert p["hbm"] == m["hbm_gbs"] and p["source"].startswith("measured")


PEAKS = {"burst": 1919.9, "sustained": 1716.3}


@pytest.mark.parametrize("clocks,kind", [
    ({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}, "burst"),           # full clock, no cap
    ({"sm_mhz": 2040.0, "sm_max_mhz": 2070.0, "reasons": []}, "burst"),           # within 3%
    ({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}, "sustained"),
    ({"sm_mhz": 1455.0, "sm_max_mhz": 2070.0, "reasons": []}, "sustained"),       # below the maximum
    ({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}, "sustained"),
])
def test_peak_follows_the_clocks_of_the_timed_region(clocks, kind):
    peak, got = bench.pick_peak(PEAKS, clocks)
    assert got == kind and peak == PEAKS[kind]


def test_roofline_fraction_reproduces_from_its_fields():
    wl = synth.WORKLOADS["wan1.3b"]
    kf = bench.kernel_flops(wl)
    r = bench.roof(kf["fine_bwd_kv"], 5.7576, PEAKS["burst"])
    assert r["tflops"] == pytest.approx(kf["fine_bwd_kv"] / 5.7576e-3 / 1e12, abs=0.01)
    assert r["frac"] == pytest.approx(r["tflops"] / PEAKS["burst"], abs=1e-4)
    assert kf["fine_bwd_kv"] == 4 * kf["dq_product"] and kf["fine_fwd"] == 2 * kf["dq_product"]
    assert kf["fine_fwd"] == bench.step_flops(wl)["fine_fwd"]
