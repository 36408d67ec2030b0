"""The bench's multi-rank bookkeeping on CPU: two gloo ranks, each timing a
different amount; both must see the slowest rank's time, and the job's
throughput counts every rank's steps against that time."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.world_max(100.0 + 50.0 * rank, "cpu")
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_world_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 150.0, 1: 150.0}


def test_single_rank_and_aggregate():
    assert bench.world_max(3.5, "cpu") == 3.5
    # 2 ranks x 10 steps in a slowest-rank time of 40 ms -> 500 steps/s
    assert bench.aggregate_steps_per_s(2, 10, 40.0) == pytest.approx(500.0)
