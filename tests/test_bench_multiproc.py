"""The benchmark's multi-rank path on CPU: two gloo ranks (no GPU).

Replicas run independent problems (no collective on the data path); the
job's time is the slowest rank's and its throughput counts every rank's
FLOPs.  Only the reduction of the timings crosses ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank            # rank 1 is the slower one
    res = bench.aggregate(local_ms, 10, 1e12, world, "cpu")
    # the reference arm does no work on ranks other than 0
    class A:
        steps, warmup = 2, 3
    skipped = bench.run_reference(A, rank, world) if rank != 0 else None
    q.put((rank, res, skipped))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, q), nprocs=2, join=True, start_method="spawn")
    out = sorted(q.get() for _ in range(2))
    for rank, (total, ms_per_step, tflops), skipped in out:
        assert total == pytest.approx(15.0)
        assert ms_per_step == pytest.approx(1.5)
        assert tflops == pytest.approx(2 * 1e12 / 1.5e-3 / 1e12)
        assert skipped is None


def test_single_rank_needs_no_process_group():
    import bench
    total, ms, tf = bench.aggregate(8.0, 4, 2e12, 1)
    assert (total, ms) == (8.0, 2.0) and tf == pytest.approx(1000.0)
