"""Multi-rank host logic of bench.py, run as two gloo ranks on the CPU.

Each rank runs the same per-GPU workload (weak scaling over independent
(b,h) units); the only exchange is the max-reduction of step times, and the
job's tokens/s counts every rank's tokens over the slowest rank's time.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.0, 5.0][rank]  # the second rank is the slow one
        m = bench.max_over_ranks(dist, ms, torch.device("cpu"))
        v = bench.job_value(world, 16384, m)
        q.put((rank, m, v))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_the_job_total():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in got:
        assert m == 5.0
        assert v == pytest.approx(2 * 16384 / 5e-3)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, 3.5, torch.device("cpu")) == 3.5
    assert bench.job_value(1, 1000, 2.0) == pytest.approx(5e5)
