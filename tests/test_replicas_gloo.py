"""The multi-GPU path is replicas only: each rank runs its own copy of the
workload and nothing crosses ranks except the timing reduction. This checks
that bookkeeping with two gloo ranks on the CPU."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per_rank_ms = [1.0 + rank, 2.0 - rank, 0.5 * (rank + 1)]
        got = bench.reduce_max(per_rank_ms, dist, device="cpu")
        out[rank] = got
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_timing_reduction_takes_max_over_two_gloo_ranks():
    world = 2
    port = 29500 + os.getpid() % 1000
    out = mp.Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert out[0] == out[1] == [2.0, 2.0, 1.0]


def test_job_throughput_is_weak_scaling_sum():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_throughput(2e12, 1, 10.0)
    assert one == pytest.approx(200.0)
    # two replicas, the slower rank sets the time
    assert bench.job_throughput(2e12, 2, 10.0) == pytest.approx(2 * one)
    assert bench.reduce_max([3.0, 1.0]) == [3.0, 1.0]
