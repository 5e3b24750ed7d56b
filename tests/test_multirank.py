"""N > 1 host logic on the CPU: two gloo ranks, no GPU.

The GEMM is not sharded: each rank runs one replica and the job's time is
the slowest rank's.  These tests check that reduction and the aggregate
throughput, and that the reference arm under torchrun prints one line from
rank 0 while the other ranks exit cleanly.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, local_ms, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.job_step_ms(local_ms[rank], 10, world)
        out[rank] = (ms, bench.job_value(2.0 * 4096 ** 3, ms, world))
    finally:
        dist.destroy_process_group()


def test_job_time_is_max_over_two_gloo_ranks():
    world, port = 2, free_port()
    local_ms = [3.0, 5.0]  # total timed ms of 10 steps on each rank
    # the manager process is started by spawn too: a fork of this process,
    # which may already run the oracle's OpenMP threads, can deadlock
    with mp.get_context("spawn").Manager() as man:
        out = man.dict()
        mp.spawn(_rank_main, args=(world, port, local_ms, out), nprocs=world, join=True)
        res = dict(out)
    assert set(res) == {0, 1}
    for r in range(world):
        ms, value = res[r]
        assert ms == pytest.approx(0.5)  # the slower rank: 5 ms / 10 steps
        # two replicas of 2*4096^3 flops every 0.5 ms
        assert value == pytest.approx(2 * 2.0 * 4096 ** 3 / 0.5e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.job_step_ms(8.0, 4, 1) == 2.0
    assert bench.job_value(1e12, 1000.0, 1) == pytest.approx(1.0)


def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "sq256_f16_f32", "--steps", "3", "--warmup", "3",
           "--ref-seconds", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["steps"] == 3 and line["warmup"] == 3
    assert line["value"] > 0 and line["e2e"]["value"] == line["value"]
    assert line["cpu_baseline"]["kind"] == "oracle"
