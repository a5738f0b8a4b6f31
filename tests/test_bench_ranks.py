"""Host logic of the multi-rank benchmark (replicas: one process per GPU):
the slowest rank's time and the whole-job rate, over two gloo ranks on the
CPU.  No GPU is used."""
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


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        seconds = 0.010 + 0.005 * rank               # rank 1 is the slower one
        slowest = bench.max_over_ranks(seconds, world)
        out[rank] = slowest
        out[world + rank] = bench.whole_job_rate(1000.0, world, slowest)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_slowest_time_and_whole_job_rate():
    world = 2
    out = torch.zeros(2 * world, dtype=torch.float64).share_memory_()
    mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == pytest.approx(0.015) and out[1] == pytest.approx(0.015)
    assert out[2] == pytest.approx(2 * 1000.0 / 0.015) and out[3] == out[2]


def test_single_rank_passes_through():
    assert bench.max_over_ranks(0.25, 1) == 0.25
    assert bench.whole_job_rate(500.0, 1, 0.5) == pytest.approx(1000.0)
