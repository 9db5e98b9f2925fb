"""Host-side logic of bench.py that decides what a run reports: the clock
summary taken from nvidia-smi samples (throttle reasons decide whether a run
is kept), the per-kernel DRAM traffic that is withdrawn once a kernel's
source changes, and the peak denominators."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sampler(lines):
    clk = bench.ClockSampler(torch.device("cpu"))
    clk.lines = lines
    return clk.summary()


def test_clock_summary_median_and_reasons():
    # clocks.sm, clocks.max.sm, power.draw, reasons bitmask, then the four
    # named reasons in ClockSampler.NAMED order.
    lines = [
        "1950, 2032, 450.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "1890, 2032, 470.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "2010, 2032, 300.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
    ]
    s = _sampler(lines)
    assert s["sm_mhz"] == 1950.0 and s["sm_mhz_min"] == 1890.0 and s["sm_max_mhz"] == 2032.0
    assert s["power_w_max"] == 470.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_thermal_and_hw_slowdown():
    lines = ["1500, 2032, 900.0, 0x48, Active, Not Active, Active, Not Active"]
    assert _sampler(lines)["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_skips_malformed_lines():
    lines = ["[N/A], 2032, 1.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage", "1900, 2032"]
    s = _sampler(lines)
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == []


def test_traffic_withdrawn_when_source_or_workload_differs(monkeypatch):
    name = "fp8_gemm_kernel"
    fname, _, workload, nbytes = bench.NCU_TRAFFIC[name]
    digest = bench._src_hash(fname)
    current = dict(bench.NCU_TRAFFIC)
    current[name] = (fname, digest, workload, nbytes)
    monkeypatch.setattr(bench, "NCU_TRAFFIC", current)
    assert bench._traffic(name, workload) == nbytes          # recorded for the current source
    assert bench._traffic(name, "some other workload") is None
    assert bench._traffic("no_such_kernel", workload) is None
    stale = dict(bench.NCU_TRAFFIC)
    stale[name] = (fname, "0" * len(digest), workload, nbytes)
    monkeypatch.setattr(bench, "NCU_TRAFFIC", stale)
    assert bench._traffic(name, workload) is None


def test_peaks_fall_back_without_measured_file(monkeypatch):
    monkeypatch.setattr(bench, "ROOT", os.path.join(ROOT, "_no_such_directory"))
    p = bench._peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6400.0 and p["bf16_tflops"] == 1800.0
    assert bench._fp8_peak(p) == pytest.approx(3600.0)
