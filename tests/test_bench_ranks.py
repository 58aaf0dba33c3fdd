"""The bench's multi-rank logic on CPU: independent replicas over gloo (world size 2).

Each rank times its own replica; the job's time is the slowest rank's, and
the reported µs per layer divides it by every layer all ranks ran.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        return sock.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 * (rank + 1)                 # rank 1 is the slow one
        total = bench.max_over_ranks(local_ms, torch.device("cpu"))
        dist.barrier()
        results[rank] = (total, bench.job_us_per_layer(total, steps=5, layers=2, world=world))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_world2():
    world = 2
    manager = mp.Manager()
    results = manager.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), results), nprocs=world, join=True)
    for rank in range(world):
        total, us = results[rank]
        assert total == 20.0                         # both ranks see the slowest rank's time
        assert us == pytest.approx(20.0 * 1e3 / (5 * 2 * world))


def test_single_process_needs_no_process_group():
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.job_us_per_layer(2.0, steps=4, layers=1, world=1) == pytest.approx(500.0)
