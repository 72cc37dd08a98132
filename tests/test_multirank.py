"""The bench's multi-rank (replicas) path on CPU: two gloo ranks on 127.0.0.1.

Each rank reports its own step time; every rank must see the max over ranks,
and the whole-job value must be world_size x per-rank work / that max."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = [2.0 + rank, 10.0 - rank, 1.5 * (rank + 1)]
        got = bench.max_over_ranks(mine, dist, "cpu")
        value = bench.replica_throughput(bench.FLOPS_STEP, world, got[0])
        results[rank] = (got, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    expect = [3.0, 10.0, 3.0]
    for r in range(world):
        got, value = res[r]
        assert got == pytest.approx(expect)
        assert value == pytest.approx(world * bench.FLOPS_STEP / (3.0e-3) / 1e12)


def test_single_rank_is_identity():
    assert bench.max_over_ranks([1.0, 2.0], None, "cpu") == [1.0, 2.0]
    assert bench.replica_throughput(2e12, 1, 1000.0) == pytest.approx(2.0)
