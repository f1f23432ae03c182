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


# ---------------------------------------------- the block-column split ----

def _shard_worker(rank, world, port, out):
    """One rank of the split on the CPU: its panel from the library's
    boundaries, its partial vector (the oracle on the matrix with every
    stored column outside the panel zeroed: exactly that panel's row and
    column terms), the gather in rank order, the rank-order sum."""
    import numpy as np
    import torch

    import oracle
    from symmetric_matrix_vector_gb300 import inputs, sharded

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    o = oracle.get()
    try:
        results = []
        for uplo in ("U", "L"):
            for n in (1, 40, 700, 1301):
                panels = sharded.split(uplo, n, world)
                every = [None] * world
                dist.all_gather_object(every, panels)
                assert all(e == panels for e in every)        # every rank: the same split
                # the panels cover the columns 0 .. n-1 exactly once, in rank order
                cols = [j for c0, c1 in panels for j in range(c0, c1)]
                assert cols == list(range(n))
                p = inputs.make_problem("s", uplo, n, lda=n + 2, alpha=1.25, beta=0.5, seed=n)

                def partial(r):
                    c0, c1 = panels[r]
                    Ar = p.A.copy()
                    outside = np.ones(n, dtype=bool)
                    outside[c0:c1] = False
                    rows = np.arange(n)
                    for j in np.nonzero(outside)[0]:      # zero the stored part of column j
                        stored = rows <= j if uplo == "U" else rows >= j
                        Ar[j, :n][stored] = 0.0
                    info, hi, _, _ = o.symv("s", uplo, n, 1.0, Ar, p.lda, p.x, 1, 0.0,
                                            np.zeros(n, np.float32), 1)
                    assert info == 0
                    return hi.astype(np.float32)

                mine = torch.from_numpy(partial(rank))
                parts = sharded.gather_in_rank_order(torch, dist, mine, world)
                # row k holds rank k's vector
                for k in range(world):
                    assert np.array_equal(parts[k].numpy(), partial(k)), (uplo, n, k)
                # the rank-order sum, merged, is the whole product (fp32 rounding)
                s = parts[0].numpy().astype(np.float32)
                for k in range(1, world):
                    s = (s + parts[k].numpy()).astype(np.float32)
                y = np.float32(1.25) * s + np.float32(0.5) * p.y
                info, hi, _, den = o.rows("s", uplo, n, 1.25, p.A, p.lda, p.x, 1, 0.5, p.y, 1,
                                          np.arange(n))
                err = float(np.max(np.abs(y.astype(np.float64) - hi) / den)) if n else 0.0
                results.append((uplo, n, err))
        out[rank] = results
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_split_columns_and_reduce_in_rank_order():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    mp.start_processes(_shard_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        for uplo, n, err in out[rank]:
            assert err <= 5e-5, (rank, uplo, n, err)


def _sum_worker(rank, world, port, out):
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.sum_over_ranks(float(rank + 1), dist, device="cpu")
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_sum_bytes_and_launches():
    """per-rank counts (bytes copied, kernels launched) add up over ranks"""
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_sum_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert out[0] == out[1] == 3.0
