"""The benchmark's multi-GPU bookkeeping, on the CPU with two gloo ranks:
every rank runs its own replica (the call does not shard), the job's time is
the slowest rank's, and the reported rate counts all replicas."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_info() == (world, rank, rank)
        ms = 1.0 + rank * 0.5                      # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, dist, device="cpu")
        rate = bench.replica_rate(world, bench.flops(1024), slowest)
        out[rank] = (slowest, rate)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        slowest, rate = out[rank]
        assert slowest == pytest.approx(1.5)
        assert rate == pytest.approx(world * 2.0 * 1024 * 1024 / 1.5e-3 / 1e9)


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(3.25, None) == 3.25
    assert bench.replica_rate(1, 2e9, 1000.0) == pytest.approx(2.0)
