"""Multi-rank host logic of bench.py on CPU: two gloo ranks.

The hot path does not shard across GPUs (each rank runs an independent
replica of the workload), so the only cross-rank steps are the barriers
around the timed region and the max over ranks of the elapsed time; the job
throughput counts every rank's bytes.
"""
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
        dist.barrier()
        # rank r "took" 10 + 5 r ms; every rank must see the slowest one
        got = bench.max_over_ranks(10.0 + 5.0 * rank, dist)
        dist.barrier()
        out[rank] = got
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_max_over_ranks_with_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_max_over_ranks_without_a_process_group_is_the_value():
    assert bench.max_over_ranks(3.25, None) == 3.25


def test_job_throughput_counts_every_rank():
    # 2 GB per step per rank at 1 ms per step: 2000 GB/s per rank
    assert bench.job_gbs(2e9, 1.0, 1) == pytest.approx(2000.0)
    assert bench.job_gbs(2e9, 1.0, 4) == pytest.approx(8000.0)
