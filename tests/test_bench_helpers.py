"""Host-side helpers of bench.py that the measurement contract rests on: the clock
summary (median SM clock under load, throttle reasons) and the rule that a recorded
DRAM traffic figure is reported only while the kernel's sources are unchanged."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _sampler_with_rows(tmp_path, rows):
    s = bench.ClockSampler(0)
    s.path = str(tmp_path / "clocks.csv")
    with open(s.path, "w") as f:
        for r in rows:
            f.write(", ".join(r) + "\n")
    s.proc = object()  # a sampler that ran
    return s


def _row(sm, mx, reasons=()):
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    flags = ["Active" if n in reasons else "Not Active" for n in names]
    return ["0", str(sm), str(mx), "900.00", "0x0", *flags]


def test_clock_summary_takes_the_median_under_load(tmp_path):
    rows = [_row(345, 2070)] * 3 + [_row(2070, 2070)] * 5 + [_row(1980, 2070, ("sw_power_cap",))] * 2
    out = _sampler_with_rows(tmp_path, rows).summary()
    assert out["samples"] == 10
    assert out["sm_max_mhz"] == 2070.0
    assert out["sm_mhz"] == 2070.0  # idle samples (below half the maximum) are left out of the median
    assert out["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_every_active_reason(tmp_path):
    rows = [_row(1500, 2070, ("hw_slowdown", "sw_thermal_slowdown"))] * 4
    out = _sampler_with_rows(tmp_path, rows).summary()
    assert out["reasons"] == ["hw_slowdown", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == 1500.0


def test_clock_summary_without_samples(tmp_path):
    out = _sampler_with_rows(tmp_path, []).summary()
    assert out["samples"] == 0 and out["sm_mhz"] is None
    none = bench.ClockSampler(0)  # never started (no nvidia-smi)
    assert none.summary()["reasons"] == ["nvidia-smi unavailable"]


def test_recorded_traffic_only_for_unchanged_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "route_sparse_gqa_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"k": ["k.cu"]})
    rec = {"k": {"bytes_per_launch": 12345, "source_hash": bench.kernel_source_hash("k")}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("k") == 12345
    assert bench.recorded_traffic("other") is None
    (csrc / "k.cu").write_text("kernel v2\n")  # the kernel changed after the capture
    assert bench.recorded_traffic("k") is None


def test_job_rate_counts_every_replica():
    # two replicas of a 1e12-FLOP step in the slowest rank's 2 ms: 1000 TFLOP/s for the job
    assert abs(bench.job_tflops(1e12, 2, 2.0) - 1000.0) < 1e-9
    assert abs(bench.job_tflops(1e12, 1, 2.0) - 500.0) < 1e-9
