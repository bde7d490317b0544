"""The benchmark's multi-rank host logic on CPU with two gloo ranks: the
slowest rank's time is what every rank reports, throughput counts every
rank's rows, and each rank draws its own batch."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(100.0 + 50.0 * rank, world)
        q.put((rank, ms, bench.rank_seed(7, rank)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [150.0, 150.0]
    assert got[0][2] != got[1][2]


def test_weak_scaling_throughput():
    assert bench.weak_scaling_throughput(8192, 1, 10, 200.0) == pytest.approx(409600.0)
    assert bench.weak_scaling_throughput(8192, 4, 10, 200.0) == pytest.approx(4 * 409600.0)
    assert bench.max_over_ranks(3.0, 1) == 3.0
