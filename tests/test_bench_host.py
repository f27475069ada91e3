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
