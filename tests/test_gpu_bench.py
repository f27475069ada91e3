"""bench.py end to end on small workloads: one JSON line with the contract's keys, and the
second precision's measurement in the same line."""
import json
import os
import subprocess
import sys

import pytest

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _check_measurement(part, steps, per_step):
    assert part["value"] > 0 and part["ms_per_step"] > 0
    roof = part["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s" and 0 < roof["frac"] == pytest.approx(
        roof["achieved"] / roof["peak"])
    assert "burst" in roof["peak_source"]
    e2e = part["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["steps"] == steps
    sb = part["step_bound"]
    assert sb["bound"] in ("tensor", "hbm") and sb["bound_ms"] == max(sb["flop_ms"], sb["byte_ms"]) > 0
    assert part["gpu_launches"] == steps * per_step


@pytest.mark.parametrize("cfg,prec,second", [("tiny", "bf16", "mxfp8"), ("qwen235b-e16", "mxfp8", "none"),
                                             ("qwen235b-e16", "bf16", "mxfp8")])
def test_bench_line(cfg, prec, second):
    need_gpu()
    r = subprocess.run([sys.executable, "bench.py", "--config", cfg, "--prec", prec, "--second-prec", second,
                        "--steps", "3", "--warmup", "3", "--no-cpu-baseline"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 3
    assert line["config"]["workload"] and "model" not in line["config"]
    per_step = {"bf16": 13, "mxfp8": 16}
    _check_measurement(line, 3, per_step[prec])
    if cfg == "tiny":                     # f = 64: outside the MXFP8 path's limits
        assert "skipped" in line["mxfp8"]
    elif second != "none":
        _check_measurement(line[second], 3, per_step[second])
        assert line[second]["config"]["precision"] == second
