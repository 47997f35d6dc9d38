"""Host-side logic of the multi-GPU bench (independent replicas, one per GPU): the
max-over-ranks reduction and the whole-job throughput, run as two gloo ranks on CPU."""
from __future__ import annotations

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.allreduce_max(1.5 + rank, world)
        val = bench.replica_value(128, world, got)
        out.put((rank, got, val))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_throughput():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, val in res:
        assert got == 2.5
        assert val == pytest.approx(128 * 2 / 2.5e-3)


def test_single_rank_passthrough():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.allreduce_max(3.25, 1) == 3.25
    assert bench.replica_value(64, 1, 0.5) == pytest.approx(64 / 0.5e-3)
