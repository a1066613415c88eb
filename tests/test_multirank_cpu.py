"""The benchmark's multi-rank logic on CPU with two gloo ranks: every rank runs
its own replica of the workload, the job's step time is the slowest rank's, the
job's throughput counts every rank's work, and only rank 0 runs the reference arm.
No data-path collective exists: the replicas exchange nothing but the timing."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 2.0 + rank  # rank 1 is the slower replica
        slowest = bench.max_over_ranks(local_ms)
        value = bench.job_tflops(slowest, world, 3 * bench.FLOP_OP)
        w, r, lr = bench.dist_env()

        class Args:
            steps, warmup, cpu_rows = 1, 0, 4
        ref = bench.run_reference(Args, w, r) if r != 0 else None  # rank 0 would time the oracle
        results[rank] = (slowest, value, w, r, lr, ref)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_job_throughput():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.start_processes(_rank_main, args=(world, port, results), nprocs=world, start_method="spawn")
        got = dict(results)
    for rank in range(world):
        slowest, value, w, r, lr, ref = got[rank]
        assert slowest == 3.0                    # the max over both ranks, seen by both
        assert (w, r, lr) == (world, rank, rank)
        assert value == pytest.approx(3 * bench.FLOP_OP * world / 3.0e-3 / 1e12)
    assert got[1][5] is None                     # rank 1 runs no reference work


def test_single_process_needs_no_process_group():
    assert bench.max_over_ranks(4.5) == 4.5
    assert bench.job_tflops(1.0, 1, 1e12) == pytest.approx(1000.0)
