"""bench.py's multi-rank rules on CPU: two gloo ranks, the slowest rank's time
sets the job's time, and the job's throughput counts every rank's tokens."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, 0, world)
        ms = [12.5, 40.0][rank]                      # rank 1 is the slow replica
        out[rank] = bench.max_over_ranks(ms, world)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 40.0


def test_single_rank_and_throughput():
    assert bench.max_over_ranks(7.25, 1) == 7.25
    # 2 ranks x 8 tokens x 100 steps in 50 ms
    assert bench.job_throughput(2, 8, 100, 50.0) == pytest.approx(32000.0)
