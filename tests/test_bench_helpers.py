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


def test_recorded_traffic_survives_comment_and_layout_edits(tmp_path, monkeypatch):
    """The recorded DRAM traffic belongs to the code: editing a comment or the layout keeps it, changing a
    token (also one inside a string literal, or one that looks like a comment marker there) drops it."""
    csrc = tmp_path / "route_sparse_gqa_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    base = 'int a = f(x);  // add one\nconst char *s = "// not a comment";\n/* block */ char c = \'"\';\n'
    (csrc / "k.cu").write_text(base)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_SOURCES", {"k": ["k.cu"]})
    rec = {"k": {"bytes_per_launch": 777, "source_hash": bench.kernel_source_hash("k")}}
    (tmp_path / "profiles" / "dram_traffic.json").write_text(json.dumps(rec))
    same = ('// a new leading comment\nint a =   f(x);\n\nconst char *s = "// not a comment";  /* more */\n'
            'char c = \'"\';  // the quote character\n')
    (csrc / "k.cu").write_text(same)
    assert bench.recorded_traffic("k") == 777
    for changed in (base.replace("f(x)", "f(y)"), base.replace('"// not a comment"', '"// changed"'),
                    base.replace("char c", "int c")):
        (csrc / "k.cu").write_text(changed)
        assert bench.recorded_traffic("k") is None


def test_job_rate_counts_every_replica():
    # two replicas of a 1e12-FLOP step in the slowest rank's 2 ms: 1000 TFLOP/s for the job
    assert abs(bench.job_tflops(1e12, 2, 2.0) - 1000.0) < 1e-9
    assert abs(bench.job_tflops(1e12, 1, 2.0) - 500.0) < 1e-9


def test_executed_pairs_against_brute_force():
    """The executed/useful pair counts of the two kernel families, recounted by brute force on a tiny case:
    tile kernels = sum over T-query tiles of ceil(distinct keys / 64) chunks; key-major kernels = sum over
    (query window, aligned 64-key chunk) of ceil(routing queries / T) groups; each chunk or group is 64 x 128
    (query-head row, key) pairs, over the routed pairs times G."""
    import numpy as np

    from route_sparse_gqa_gb300 import workloads as W

    w = W.Workload(99, "t", 1, 70, 300, 16, 2, 256, 12, np.int32, 0.0625, "t")
    rng = np.random.default_rng(3)
    ids = np.full((1, 70, 12), -1, np.int32)
    counts = np.zeros((1, 70), np.int32)
    for q in range(70):
        n = int(rng.integers(0, 13))
        ids[0, q, :n] = np.sort(rng.choice(300, size=n, replace=False))
        counts[0, q] = n
    got = bench.executed_pairs(w, ids, counts)
    G, T = 8, 16
    tiles = sum(-(-len(set(ids[0, t:t + T][ids[0, t:t + T] >= 0].tolist())) // 64) for t in range(0, 70, T))
    # one window covers all 70 rows here (the window is thousands of rows)
    per_chunk = {}
    for q in range(70):
        for c in set((ids[0, q, :counts[0, q]] // 64).tolist()):
            per_chunk[c] = per_chunk.get(c, 0) + 1
    groups = sum(-(-n // T) for n in per_chunk.values())
    useful = int(counts.sum()) * G
    assert got["tile_chunks"] == tiles and got["keymajor_groups"] == groups
    assert abs(got["tile_over_useful"] - round(tiles * 64 * 128 / useful, 3)) < 1e-9
    assert abs(got["keymajor_over_useful"] - round(groups * 64 * 128 / useful, 3)) < 1e-9
