"""bench.py's JSON line, as the benchmark harness reads it: the forward
layer, the backward (--backward) and the oracle arm (--impl reference), on
the small layer so that each run takes seconds."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"),
                          "--workload", "small", *args],
                         capture_output=True, text=True, timeout=900,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-3000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, out.stdout[-2000:]
    return json.loads(lines[0])


def check_common(j, steps, warmup):
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup",
                "ms_per_step", "higher_is_better", "scaling", "vs_baseline",
                "dtype", "data", "config"):
        assert key in j, key
    assert j["value"] > 0 and j["ms_per_step"] > 0
    assert j["unit"] == "tokens/s" and j["higher_is_better"] is True
    assert j["n_gpus"] == 1 and j["steps"] == steps and j["warmup"] == warmup
    assert j["scaling"] == "weak" and j["vs_baseline"] is None
    assert j["config"]["workload"]


def check_roofline(j):
    r = j["roofline"]
    for key in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert key in r, key
    assert r["bound"] in ("hbm", "tensor")
    assert r["achieved"] > 0 and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"], rel=1e-2)


def check_e2e(j):
    e = j["e2e"]
    assert e["value"] > 0 and e["unit"] == j["unit"]
    assert e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0


def test_forward_line():
    j = run_bench("--steps", "3", "--warmup", "3", "--no-cpu-baseline")
    check_common(j, 3, 3)
    check_roofline(j)
    check_e2e(j)
    assert j["gpu_launches"] > 0
    assert j["dtype"] == "bf16"


def test_backward_line():
    j = run_bench("--backward", "--steps", "2", "--warmup", "3")
    check_common(j, 2, 3)
    check_roofline(j)
    check_e2e(j)
    assert j["gpu_launches"] > 0
    cb = j["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["cores"] >= 1
    assert "backward" in j["metric"]


def test_reference_arm_line():
    j = run_bench("--impl", "reference", "--steps", "1", "--warmup", "0")
    assert j["impl"] == "reference"
    check_common(j, 1, 0)
    assert j["cpu_baseline"]["kind"] == "oracle"
    assert j["e2e"]["h2d_bytes_per_step"] == 0
