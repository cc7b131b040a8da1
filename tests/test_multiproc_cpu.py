"""The multi-process side of bench.py on CPU ranks (gloo, world size 2).

Decode shards by independent work: every rank runs its own replica of the
workload and the only exchange is the timing reduction at the end (max of the
per-rank seconds, sum of the per-rank units).  These tests run that reduction
on two gloo ranks and check the reference arm's rank handling.
"""

import io
import os
import socket
import sys
from contextlib import redirect_stdout

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


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    bench.barrier()
    # rank r processed r + 1 units in 0.5 + r seconds
    value, slowest, n = bench.aggregate(rank + 1.0, 0.5 + rank)
    mx = bench.reduce_max(10.0 - rank)
    out[rank] = (value, slowest, n, mx)
    dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    # whole-job throughput = units summed over ranks / the slowest rank's time
    for rank in range(world):
        value, slowest, n, mx = out[rank]
        assert n == world
        assert slowest == pytest.approx(1.5)
        assert value == pytest.approx((1.0 + 2.0) / 1.5)
        assert mx == pytest.approx(10.0)


def test_single_process_aggregate_is_the_identity():
    import bench
    assert not dist.is_initialized()
    value, slowest, n = bench.aggregate(6.0, 2.0)
    assert (value, slowest, n) == (3.0, 2.0, 1)
    assert bench.reduce_max(4.5) == 4.5


def test_reference_arm_prints_only_on_rank_zero(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"])
    assert rc == 0
    assert buf.getvalue() == ""
