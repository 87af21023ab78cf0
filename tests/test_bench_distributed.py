"""The bench's multi-rank plumbing on CPU: two gloo ranks, each with its own
step time; the reported time is the slowest rank's and the throughput counts
every rank's layer step (weak scaling: ranks share no data on this path)."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 2.0 + rank  # rank 1 is slower
        out[rank] = bench.reduce_max_over_ranks(ms, world)
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1] == 3.0
    one = bench.whole_job_tflops(3.0, 1)
    assert bench.whole_job_tflops(3.0, world) == pytest.approx(2 * one)
    assert one == pytest.approx(6 * 8192 * 5120 * 20480 / 3e-3 / 1e12)


def test_single_rank_is_identity():
    assert bench.reduce_max_over_ranks(1.25, 1) == 1.25
