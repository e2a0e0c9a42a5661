"""Host logic of bench.py on CPU: the clock record it attaches to a run (median
SM clock under load, throttle reasons that reject a run), the peaks it divides
by, and the work it counts per step."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from memory_efficient_cnn_gb300 import workloads as wl  # noqa: E402


class _DoneProcess:
    """Stands in for the finished nvidia-smi process."""

    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _clocks_from(tmp_path, lines):
    s = bench.ClockSampler(0)
    s.out = str(tmp_path / "clocks.csv")
    with open(s.out, "w") as f:
        f.write("\n".join(lines) + "\n")
    s.proc = _DoneProcess()
    return s.stop()


def test_clock_record_takes_the_median_under_load(tmp_path, monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda _s: None)
    idle = "0, 345, 2070, 150.0, 0x0, Not Active, Not Active, Not Active, Not Active"
    busy = ["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2055, 2070, 950.0, 0x0, Not Active, Not Active, Not Active, Not Active",
            "0, 2070, 2070, 980.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    rec = _clocks_from(tmp_path, [idle] + busy + [idle])
    assert rec["sm_mhz"] == 2070.0  # the idle samples (below half the max) are left out
    assert rec["sm_max_mhz"] == 2070.0
    assert rec["reasons"] == [] and rec["samples"] == 5
    assert not os.path.exists(tmp_path / "clocks.csv")


def test_clock_record_names_the_throttle_reasons(tmp_path, monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda _s: None)
    rows = ["0, 1800, 2070, 1400.0, 0x4, Not Active, Not Active, Not Active, Active",
            "0, 1500, 2070, 1400.0, 0x48, Not Active, Active, Not Active, Active"]
    rec = _clocks_from(tmp_path, rows)
    assert rec["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]
    assert rec["sm_mhz"] == 1650.0


def test_clock_record_without_samples(tmp_path, monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda _s: None)
    rec = _clocks_from(tmp_path, ["garbage"])
    assert rec["sm_mhz"] is None and rec["reasons"] == ["no samples"]
    s = bench.ClockSampler(0)
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_peaks_come_from_the_measured_file_else_the_fallback(tmp_path, monkeypatch):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps(
        {"hbm_gbs": 6803.8, "bf16_tflops": 1942.5, "bf16_tflops_sustained": 1699.9, "sm_max_mhz": 2070}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench._peaks()
    assert p["source"] == "measured" and p["hbm_gbs"] == 6803.8 and p["bf16_tflops"] == 1942.5
    monkeypatch.setattr(bench, "ROOT", str(tmp_path / "missing"))
    p = bench._peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0 and p["bf16_tflops"] == 1900.0


def test_step_work_counts():
    # cv1: 2 * N * C_o * H_o * W_o * C_i * H_f * W_f with H_o = W_o = 55
    assert bench.conv_flops(wl.CV1) == 2.0 * 128 * 96 * 55 * 55 * 3 * 11 * 11
    assert bench.conv_flops(wl.CV1) == pytest.approx(26.99e9, rel=1e-3)
    # padding 1 keeps the 56x56 extent of the 3x3 sweep layer
    assert bench.conv_flops(wl.SAME_3x3) == 2.0 * 64 * 128 * 56 * 56 * 128 * 9
    assert "padding 1x1" in bench.workload_str(wl.SAME_3x3)
    assert bench.workload_str(wl.CV1).startswith("cv1: N=128, C_i=3, 227x227, C_o=96, 11x11, stride 4x4")
    assert bench.job_tflops(4, 1e12, 1.0) == pytest.approx(4000.0)
