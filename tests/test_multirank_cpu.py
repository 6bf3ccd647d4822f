"""The N > 1 path of bench.py on the CPU: two gloo ranks, each an independent
replica (no data-path collective); the timing takes the slowest rank and the
throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms)
        out[rank] = slowest
        out[world + rank] = bench.job_throughput(4096, world, 20, slowest)
        # replicas draw their own inputs: rank-dependent seeds give different routings
        import workloads
        w = workloads.scaled(workloads.WORKLOADS["tiny"], T=64)
        idx, _ = workloads.router(w, seed=rank)
        out[2 * world + rank] = float(idx.astype("float64").sum())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_slowest_time_and_job_throughput():
    world = 2
    out = torch.zeros(3 * world, dtype=torch.float64).share_memory_()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0].item() == out[1].item() == 15.0
    assert out[2].item() == out[3].item() == pytest.approx(4096 * 2 * 20 / 0.015)
    assert out[4].item() != out[5].item()


def test_single_process_is_identity():
    import bench

    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.job_throughput(100, 1, 10, 1000.0) == 1000.0
