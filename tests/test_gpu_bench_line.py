"""The measurement line bench.py prints, checked on small workloads.

Runs bench.py in a subprocess as a user would (one workload, a few steps) and
checks the keys and the arithmetic of its JSON line: the metric and its unit,
the timing fields, the roofline object of the dominant kernel (achieved / peak
= frac), the end-to-end figure with the bytes it moved, the launch count, the
clock record, and the oracle's CPU baseline.
"""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench_line(*args):
    env = dict(os.environ)
    env.pop("BIGEMM_PLAN_CACHE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


def check_common(d, workload, steps):
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches",
              "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["warmup"] >= 3
    assert d["scaling"] == "weak" and d["higher_is_better"] is True and d["data"] == "synthetic"
    assert d["config"]["workload"].startswith(workload)
    assert d["value"] > 0 and d["ms_per_step"] > 0
    rf = d["roofline"]
    assert rf["bound"] in ("hbm", "tensor", "alu") and rf["unit"] in ("GB/s", "TFLOP/s")
    assert rf["peak"] > 0 and rf["achieved"] > 0
    assert abs(rf["frac"] - rf["achieved"] / rf["peak"]) < 1e-6 * max(1.0, rf["frac"])
    assert 0 < rf["frac"] < 1.5, "a roofline fraction far above 1 means the kernel is not doing the work"
    e = d["e2e"]
    assert e["unit"] == d["unit"] and 0 < e["value"] <= d["value"] * 1.05
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= steps
    ck = d["clocks"]
    assert ck["sm_mhz"] > 0 and ck["sm_max_mhz"] > 0 and isinstance(ck["reasons"], list)


def test_bench_line_conv_workload():
    d = bench_line("--only", "--workload", "resnet_last", "--steps", "4", "--warmup", "3")
    check_common(d, "resnet_last", 4)
    assert d["unit"] == "TFLOP/s" and d["dtype"] == "tf32"
    assert d["per_layer"] and all(l["us"] > 0 for l in d["per_layer"])
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] > 0 and cb["sample"]
    # the timed work is the layer's FLOP over the measured step time
    flop = 2 * 1 * 512 * 7 * 7 * 512 * 9
    assert abs(d["value"] - flop / (d["ms_per_step"] * 1e-3) / 1e12) < 1e-6 * d["value"]


def test_bench_line_broadcast():
    d = bench_line("--only", "--workload", "bcast", "--steps", "4", "--warmup", "3", "--no-cpu-baseline")
    check_common(d, "bcast", 4)
    assert d["unit"] == "GB/s" and d["roofline"]["bound"] == "hbm"
    assert set(d["bcast_ab"]) >= {"exp", "rsqrt"} and d["bcast_general"]
    assert "cpu_baseline" not in d
