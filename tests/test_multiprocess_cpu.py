"""The benchmark's N > 1 host path on CPU: two gloo ranks, no GPU.

Each rank runs its own replica of the workload (the read shards along
tokens with no exchange), times itself, and the job's number is all ranks'
tokens over the slowest rank's time.  Only that timing reduction and the
barrier cross ranks."""
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


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    bench.dist_init(world, "gloo")
    bench.barrier(world)
    elapsed = 100.0 + 50.0 * rank                  # rank 1 is the slow one
    mx = bench.max_over_ranks(elapsed, world, "cpu")
    value = bench.aggregate(1000, 10, world, mx)
    bench.barrier(world)
    q.put((rank, mx, value))
    dist.destroy_process_group()


def test_two_rank_timing_reduction_and_aggregate():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, value in res:
        assert mx == 150.0
        assert value == pytest.approx(1000 * 10 * 2 / 0.150)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.aggregate(32768, 100, 1, 1000.0) == pytest.approx(3276800.0)
