"""Host-side parts of bench.py (no GPU): the committed traffic record is bound
to the kernel source it was measured on, the peak comes from the measured
file, the spread helper, and the CPU baseline's fields."""
import json
import os

import pytest

import bench
import spec_inputs as si


def test_traffic_record_matches_the_committed_source():
    rec = bench.traffic_record(si.C5.name)
    if rec is None:   # bench.py then reports traffic null until the next capture
        pytest.skip("the committed traffic record predates the current kernel source")
    assert rec["source_sha256_16"] == bench.source_sha()
    # DRAM traffic of a launch is the algorithmic bytes plus a small workspace share
    assert 1.0 <= rec["dram_bytes_per_launch"] / rec["algorithmic_bytes_per_launch"] < 1.02
    assert rec["algorithmic_bytes_per_launch"] == si.C5.scaled(batch=rec["batch"]).logit_bytes


def test_traffic_record_rejects_another_source(monkeypatch, tmp_path):
    other = tmp_path / "other.cu"
    other.write_text("// not the kernel\n")
    monkeypatch.setattr(bench, "CU_SOURCE", str(other))
    assert bench.traffic_record(si.C5.name) is None


def test_peak_is_the_measured_copy_rate():
    value, kind = bench.peaks()
    path = os.path.join(bench.ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        assert kind == "measured" and value == float(json.load(open(path))["hbm_gbs"])
    else:
        assert kind == "fallback" and value == 6800.0


def test_spread():
    s = bench.spread_us([1.0, 2.0, 3.0, 4.0, 5.0])
    assert s["n"] == 5 and s["p50"] == 3000.0 and s["p10"] < s["p50"] < s["p90"]


def test_cpu_baseline_fields():
    pytest.importorskip("numpy")
    r = bench.cpu_baseline(si.TINY.scaled(batch=8, vocab=64), target_seconds=0.2)
    assert r["kind"] == "oracle" and r["unit"] == bench.UNIT and r["cores"] >= 1 and r["value"] > 0
    assert r["single_thread"]["value"] > 0 and "chains" in r["sample"]
