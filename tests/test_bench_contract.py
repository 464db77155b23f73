"""bench.py's contract pieces that run without a GPU: the reference arm (the
oracle timed on the host cores) prints one JSON line with the keys the
benchmark contract names, and the roofline helpers compute what they say."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_reference_arm_json_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["steps"] == 1 and d["warmup"] == 0 and d["n_gpus"] == 1
    assert d["config"]["workload"] == bench.MAIN
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], cwd=ROOT, capture_output=True, text=True,
                         timeout=300, env=env)
    assert out.returncode == 0 and "{" not in out.stdout


def test_roofline_obj():
    r = bench.roofline_obj("hbm", 3242.75, 6485.5, "GB/s", 1.0e9)
    assert r == {"bound": "hbm", "achieved": 3242.75, "peak": 6485.5, "unit": "GB/s",
                 "frac": 0.5, "traffic": 1.0e9}


def test_per_layer_roofline():
    pl = {"swa_ms": 2.0, "ga_ms": 100.0, "swa_bytes": 6.4855e9, "ga_flops": 8.7565e13}
    r = bench.per_layer_roofline(pl, {"hbm_gbs": 6485.5, "bf16_tflops": 1751.3})
    assert r["swa_gbs"] == pytest.approx(3242.75)
    assert r["swa_frac_hbm"] == pytest.approx(0.5)
    assert r["ga_tflops"] == pytest.approx(875.65)
    assert r["ga_frac_tensor"] == pytest.approx(0.5)


def test_traffic_table_scales_and_goes_stale(monkeypatch):
    # a current entry scales with the units processed
    b = bench.traffic_for("band", 32768)
    if b is not None:
        assert bench.traffic_for("band", 4 * 32768) == pytest.approx(4 * b)
    # an entry whose kernel sources changed since the capture reports nothing
    monkeypatch.setattr(bench, "kernel_hash", lambda kernel: "0" * 64)
    assert bench.traffic_for("band", 32768) is None
    assert bench.traffic_for("no_such_entry", 1) is None
