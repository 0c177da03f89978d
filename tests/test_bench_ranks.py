"""Multi-rank host logic of bench.py on the CPU: two gloo ranks on 127.0.0.1.

The layer does not shard (one replica per GPU, no collective on the data path), so
the only cross-rank steps are the timing ones: every rank's time is replaced by the
slowest rank's, and the job's rate counts every rank's units over that time.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.slowest_rank_ms(1.0 + 2.0 * rank, world, "cpu")    # rank 0: 1 ms, rank 1: 3 ms
        q.put((rank, ms, bench.job_throughput(world, 100.0, ms)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_time_and_job_throughput_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, ms, rate in got:
        assert ms == 3.0                                   # both ranks see the slowest time
        assert rate == pytest.approx(2 * 100.0 / 3e-3)     # both ranks' units over it


def test_one_rank_keeps_its_own_time():
    assert bench.slowest_rank_ms(2.5, 1, "cpu") == 2.5
    assert bench.job_throughput(1, 10.0, 2.0) == pytest.approx(5000.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the oracle arm is rank 0's alone: another rank exits 0, prints nothing."""
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
