"""bench.py's JSON line on the GPU (the small workload): every key of the
contract is present, the timed numbers are consistent with each other, and
the roofline fraction is achieved / peak."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_json_line_small():
    cmd = [sys.executable, "bench.py", "--workload", "small", "--steps", "5", "--warmup", "3",
           "--no-cpu-baseline", "--produce-steps", "2", "--other-configs", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches", "clocks", "prepare", "produce"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["warmup"] == 3
    assert d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["ms_per_step"] > 0
    # value = work per step / step time
    gflop = d["config"]["gflop_per_step"]
    assert abs(d["value"] - gflop / d["ms_per_step"]) <= 1e-6 * d["value"]
    rf = d["roofline"]
    assert rf["bound"] == "tensor" and rf["peak"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-9
    assert rf["ms_per_launch"] <= d["ms_per_step"]
    assert 0 < rf["sfu"]["frac"] < 2
    e2e = d["e2e"]
    assert e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["ms_per_step"] > 0
    assert d["gpu_launches"] == 3 * d["steps"]
    assert d["produce"]["ms_per_call"] > 0 and 0 < d["produce"]["frac"] < 2
    assert "sm_mhz" in d["clocks"]
    # step bins cover the timed steps in order
    bins = d["step_bins"]
    assert bins[0]["steps"][0] == 0 and bins[-1]["steps"][1] == d["steps"]
    assert all(b["forward_ms"] > 0 for b in bins)
    # the other workloads' lines
    t = d["configs"]["tiny"]
    assert t["ms_per_forward"] > 0 and t["ms_per_prepare"] > 0
    assert t["ms_per_forward"] + t["ms_per_prepare"] <= t["ms_per_step"] * 1.001
    assert abs(t["roofline"]["frac"] - t["roofline"]["achieved"] / t["roofline"]["peak"]) < 1e-9
    assert "sm_mhz" in t["clocks"]
