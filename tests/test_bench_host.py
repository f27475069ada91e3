"""Host-side pieces of bench.py, without a GPU: the clock summary from nvidia-smi output,
the recorded-traffic lookup, the reference-arm sample size and flag checks."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

# canned `nvidia-smi --query-gpu=<ClockSampler.FIELDS> --format=csv,noheader,nounits` lines
SMI = """2026/12/03 00:00:00.000, GPU-abc, 2070, 2070, 300.5, Not Active, Not Active, Not Active, Not Active
2026/12/03 00:00:00.100, GPU-abc, 1800, 2070, 1390.0, Not Active, Not Active, Not Active, Active
2026/12/03 00:00:00.150, GPU-abc, 1850, 2070, 1385.0, Not Active, Not Active, Not Active, Active
2026/12/03 00:00:00.200, GPU-def, 900, 2070, 200.0, Active, Not Active, Not Active, Not Active
2026/12/03 00:00:00.400, GPU-abc, 2070, 2070, 310.0, Not Active, Not Active, Not Active, Not Active
"""


def _t(hms):
    import datetime
    return datetime.datetime.strptime("2026/12/03 " + hms, "%Y/%m/%d %H:%M:%S.%f").timestamp()


def test_clock_summary_keeps_this_gpu_inside_the_timed_window():
    c = bench.ClockSampler.summarise(SMI, "abc", _t("00:00:00.050"), _t("00:00:00.300"))
    assert c["samples"] == 2 and c["in_timed_window"]
    assert c["sm_mhz"] == 1825.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]  # the other GPU's hw_slowdown is not ours


def test_clock_summary_without_window_uses_every_sample_of_this_gpu():
    c = bench.ClockSampler.summarise(SMI, "abc")
    assert c["samples"] == 4 and not c["in_timed_window"]
    assert c["reasons"] == ["sw_power_cap"]


def test_recorded_traffic_follows_the_kernel_sources():
    for prec in ("bf16", "mxfp8"):
        h = bench.source_hash(prec)
        assert len(h) == 16 and h == bench.source_hash(prec)
    assert bench.read_traffic("bf16:no-such-workload:gate_up") is None
    lines = [ln.split() for ln in open(os.path.join(ROOT, "profiles", "dram_traffic.txt")) if not ln.startswith("#")]
    for key, nbytes, h, *_ in lines:
        assert float(nbytes) > 0
        if h == bench.source_hash(key.split(":")[0]):
            assert bench.read_traffic(key) == float(nbytes)


def test_oracle_sample_is_smaller_for_mxfp8():
    class A:
        ref_tokens = 32
        prec = "bf16"
    assert bench.oracle_chunk(A) == 32
    A.prec = "mxfp8"
    assert bench.oracle_chunk(A) == 4


def test_weights_cached_needs_mxfp8():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--weights-cached"], capture_output=True,
                       text=True, cwd=ROOT)
    assert r.returncode != 0 and "--weights-cached applies to --prec mxfp8" in r.stderr


def _dense_cfg(**kw):
    from dropless_mixture_experts_warp_gb300 import synth
    base = dict(T=128, d=128, f=64, E=1, k=1, score="softmax", bias="zero", seed=1)
    base.update(kw)
    return synth.MoEConfig("hand", **base)


def test_step_bytes_of_a_small_dense_step_by_hand():
    # T = R = 128 rows, d = 128, f = 64, one expert; bf16 elements are 2 bytes:
    # route 128*1*4 + 128*1*8 = 1536; dispatch 2 * 128*128*2 = 65536;
    # gate/up: x 32768 + W_gu (128x128) 32768 + G|U 32768 + h 16384 = 114688;
    # down: h 16384 + W_d 16384 + y 32768 = 65536;
    # down dgrad: dY rows 32768 + W_d 16384 + G|U 32768 + dG|dU 32768 = 114688;
    # down wgrad: 32768 + 16384 + dW_d 16384 = 65536;
    # gate/up dgrad: dG|dU 32768 + W_gu 32768 + dX rows 32768 = 98304;
    # gate/up wgrad: 32768 + 32768 + dW_gu 32768 = 98304;
    # combine, combine backward, un-permute 65536 each; router backward 1024 + 1536 = 2560
    cfg = _dense_cfg()
    assert bench.step_bytes(cfg, "bf16") == 1536 + 65536 + 557056 + 3 * 65536 + 2560


def test_step_bytes_weight_quantisation_term():
    # MXFP8: cached weights save reading both bf16 weights once (2 bytes an element) and
    # writing their codes in two orientations (1 + 1/32 bytes an element each)
    cfg = _dense_cfg()
    w = 3 * 128 * 64
    saved = bench.step_bytes(cfg, "mxfp8") - bench.step_bytes(cfg, "mxfp8", weights_cached=True)
    assert saved == w * 2 + 2 * w * (1 + 1 / 32)
    sh = _dense_cfg(f_shared=64)
    saved_sh = bench.step_bytes(sh, "mxfp8") - bench.step_bytes(sh, "mxfp8", weights_cached=True)
    assert saved_sh == 2 * saved                       # the shared expert's weights too


def test_step_bound_picks_the_slower_roof():
    from dropless_mixture_experts_warp_gb300 import synth
    mix = synth.CONFIGS["mixtral"]
    b = bench.step_bound(mix, "bf16", False, 10.0, 1719.5, 6764.0)
    assert b["bound"] == "tensor" and b["bound_ms"] == b["flop_ms"] > b["byte_ms"]
    assert abs(b["flop_ms"] - mix.flops_fwd_bwd() / 1719.5e12 * 1e3) < 1e-12
    assert abs(b["frac"] - b["bound_ms"] / 10.0) < 1e-12
    probe = synth.CONFIGS["hbm-probe"]
    b = bench.step_bound(probe, "bf16", False, 2.0, 1719.5, 6764.0)
    assert b["bound"] == "hbm" and b["bound_ms"] == b["byte_ms"] == b["bytes"] / 6764e9 * 1e3
    for cfg in synth.CONFIGS.values():
        for prec in ("bf16", "mxfp8"):
            assert bench.step_bytes(cfg, prec) > 0


def test_reference_arm_line_on_the_tiny_workload():
    """--impl reference times the CPU oracle (no GPU involved) and prints one line with the
    contract's keys, its own cpu_baseline and an e2e without host copies."""
    import json
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "2", "--warmup", "3"], capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    for key in ("metric", "value", "unit", "n_gpus", "ms_per_step", "higher_is_better", "config", "cpu_baseline",
                "e2e"):
        assert key in line, key
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] > 0 and cb["cores"] >= 1
    from dropless_mixture_experts_warp_gb300 import synth
    assert abs(cb["extrapolated_full_step_s"] - synth.CONFIGS["tiny"].flops_fwd_bwd() / (cb["value"] * 1e12)) < 1e-9
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
