"""The multi-rank arithmetic of bench.py on CPU: two gloo ranks, each with its
own time, report the slowest rank's time and the whole job's rows per second;
each rank samples its own seeded batch (replicas over rows)."""
from __future__ import annotations

import os
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        slowest, rate = bench.whole_job_rate(1.0 + rank, 100, world, torch.device("cpu"))
        w = bench.make_workload("tiny", rank)
        out[rank] = (slowest, rate, int(w.seed[0]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world = 2
    port = 29500 + os.getpid() % 2000
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    for r in range(world):
        slowest, rate, _ = res[r]
        assert slowest == 2.0
        assert rate == pytest.approx(100 * world / 2.0)
    assert res[0][2] != res[1][2], "each rank samples its own batch"
