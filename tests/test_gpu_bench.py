"""bench.py end to end on the tiny workload: one JSON line with the contract's keys."""
import json
import os
import subprocess
import sys

import pytest

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("prec", ["bf16", "mxfp8"])
def test_bench_line(prec):
    need_gpu()
    cfg = "tiny" if prec == "bf16" else "qwen235b-e16"
    r = subprocess.run([sys.executable, "bench.py", "--config", cfg, "--prec", prec, "--steps", "3", "--warmup", "3",
                        "--no-cpu-baseline"], cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["value"] > 0 and line["ms_per_step"] > 0
    assert line["config"]["workload"] and "model" not in line["config"]
    roof = line["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and 0 < roof["frac"] == pytest.approx(
        roof["achieved"] / roof["peak"])
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    sb = line["step_bound"]
    assert sb["bound"] in ("tensor", "hbm") and sb["bound_ms"] == max(sb["flop_ms"], sb["byte_ms"]) > 0
    per_step = 13 if prec == "bf16" else 16
    assert line["gpu_launches"] == 3 * per_step
