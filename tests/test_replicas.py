"""The N-GPU bench path is N independent replicas: the job's step time is the slowest
rank's and its rate counts every replica's work.  Exercised with two gloo ranks on CPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [10.0 + 5.0 * rank, 3.0 - rank]          # rank 1 is slower on the first value only
    got = bench.reduce_max(local, dist, torch.device("cpu"))
    out[rank] = got
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_replica_sets_the_time_and_all_work_counts():
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == [15.0, 3.0]
    import bench
    # two replicas of 17.32 TFLOP each in 15 ms
    assert bench.job_rate(2, 17.32e12, 15.0) == pytest.approx(2 * 17.32e12 / 15e-3 / 1e12)


def test_single_process_is_the_identity():
    import bench
    assert bench.reduce_max([1.5, 2.5], None, None) == [1.5, 2.5]


def _run_bench(args, env_extra):
    import subprocess
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, capture_output=True, text=True,
                          env=env, timeout=600, cwd=ROOT)


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0"],
                   {"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_line():
    import json
    r = _run_bench(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1"],
                   {"RANK": "0", "WORLD_SIZE": "1"})
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
