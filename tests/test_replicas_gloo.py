"""The multi-rank path of the benchmark on CPU: two ``gloo`` ranks, each timing
its own replica, agree on the slowest rank's time and report the job's
throughput as all ranks' steps over that time."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, ms_per_rank, steps, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms_max = bench.max_over_ranks(ms_per_rank[rank], world, "cpu")
        out[rank] = (ms_max, bench.replica_throughput(steps, ms_max, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    world, steps = 2, 50
    ms_per_rank = [80.0, 125.0]
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank, args=(world, _free_port(), ms_per_rank, steps, out), nprocs=world, join=True,
                       start_method="spawn")
    for rank in range(world):
        ms_max, value = out[rank]
        assert ms_max == 125.0
        assert value == pytest.approx(world * steps / 0.125)


def test_one_rank_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.replica_throughput(10, 20.0, 1) == pytest.approx(500.0)
