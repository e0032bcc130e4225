"""The benchmark's JSON line, as its readers see it: the default invocation (every extra included) must
end its stdout with one compact JSON object carrying the contract keys, short enough that a reader
keeping only the last 1500 characters of stdout still holds all of it."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
MAX_LINE_BYTES = 1400


def check_line(d, steps):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks", "e2e", "cpu_baseline"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] >= 3 and d["higher_is_better"] is False
    assert d["value"] > 0 and d["gpu_launches"] == steps * 20
    assert "workload" in d["config"] and "T=128" in d["config"]["workload"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["unit"] == "GB/s" and 0 < rf["frac"] < 1.5
    assert abs(rf["achieved"] / rf["peak"] - rf["frac"]) < 1e-3
    assert rf["algorithmic_bytes_per_launch"] == 61_378_560
    assert "traffic" in rf
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(d["clocks"])
    e = d["e2e"]
    assert e["unit"] == d["unit"] and e["value"] > d["value"]
    assert e["h2d_bytes_per_step"] > 50_000_000 and e["d2h_bytes_per_step"] == 2 * 128 * 6144 * 2
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["unit"] == d["unit"] and cb["sample"]


@pytest.mark.gpu
def test_default_bench_line_is_last_compact_and_complete(tmp_path):
    extras = tmp_path / "extras.json"
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3",
                        "--cpu-budget", "1", "--extras-out", str(extras)],
                       capture_output=True, text=True, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    last = r.stdout.rstrip("\n").split("\n")[-1]
    assert len(last.encode()) <= MAX_LINE_BYTES, len(last.encode())
    d = json.loads(last)
    check_line(d, 5)
    s = d["summary"]
    assert s["T1_us"] > 0 and s["T1_x_floor"] >= 1.0 and s["T16_us"] > 0
    assert 0.3 < s["frac_H7168_T16384_bf16"] < 1.5
    x = json.load(open(extras))
    assert {"sweep_l2_warm", "configs", "finalize_only_and_unfused_l2_warm", "launch_floor_us"} <= set(x)
    # tiny 1 + masked 3 top-k x 2 act x 2 R x 2 scale dtypes x 4 T + high top-k 3 x 6 + bandwidth 2 H x 3 T x 4 outputs
    assert len(x["configs"]) == 1 + 96 + 18 + 24


@pytest.mark.gpu
def test_headline_only_bench_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "5", "--warmup", "3",
                        "--no-extras", "--cpu-budget", "1"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    assert len(lines[0].encode()) <= MAX_LINE_BYTES
    check_line(json.loads(lines[0]), 5)
