"""The benchmark's multi-rank arithmetic on CPU (gloo, world size 2): each rank
runs its own token stream (replicas, no data-path collective); the job's time
per step is the slowest rank's, and throughput counts every rank's tokens."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, local_ms, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        ms = bench.job_time(local_ms[rank], world, torch.device("cpu"))
        out[rank] = (ms, bench.whole_job_us_per_token(ms, 256, world))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, local_ms = 2, [4.0, 6.5]
    port = 29500 + (os.getpid() % 1000)
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, local_ms, out), nprocs=world, start_method="spawn")
        res = dict(out)
    for r in range(world):
        ms, us = res[r]
        assert ms == pytest.approx(6.5)
        assert us == pytest.approx(6.5 * 1000.0 / (256 * world))


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.job_time(3.25, 1, torch.device("cpu")) == 3.25
    assert bench.whole_job_us_per_token(3.25, 256, 1) == pytest.approx(3.25 * 1000.0 / 256)
