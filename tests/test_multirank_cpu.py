"""The multi-rank host logic of bench.py on CPU: two gloo ranks, no GPU.

Each rank of a multi-GPU run times its own replica; the reported time is the slowest rank's and
the throughput sums every rank's cached tokens over that time (weak scaling, no data-path
collective).
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        local_ms = [265.0, 271.5][rank]          # each replica's own timed region
        slowest = bench.max_over_ranks(local_ms, "cpu")
        value = bench.weak_scaling_value(32768.0, world, slowest)
        out[rank] = torch.tensor([slowest, value], dtype=torch.float64)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    for r in range(world):
        slowest, value = out[r].tolist()
        assert slowest == 271.5
        assert value == pytest.approx(2 * 32768.0 / 0.2715)


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(3.0, "cpu") == 3.0
    assert bench.weak_scaling_value(10.0, 1, 1000.0) == pytest.approx(10.0)
