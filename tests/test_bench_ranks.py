"""The bench's multi-process path (one replica per GPU) on CPU: two gloo ranks time different
steps; every rank must see the slowest rank's time, and the whole-job throughput counts every
rank's tokens over that time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                 # rank 1 is slower
        slowest = bench.max_over_ranks(mine, dist, "cpu")
        q.put((rank, slowest, bench.job_throughput(1000, world, slowest / 4)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_all_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in got:
        assert slowest == 15.0
        assert value == pytest.approx(2 * 1000 / (3.75e-3))


def test_single_process_is_identity():
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.job_throughput(1000, 1, 50.0) == pytest.approx(20000.0)
