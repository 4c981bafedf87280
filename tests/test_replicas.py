"""Multi-process (world size 2, gloo, CPU) test of the replica logic bench.py
uses when it runs one process per GPU: each rank draws its own workload copy,
the slowest rank sets the step time, and the value is the whole job's
throughput."""
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
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    times = [10.0 + 5 * rank, 3.0 - rank]
    red = bench.max_over_ranks(times, dist)
    seeds = [None] * world
    dist.all_gather_object(seeds, bench.replica_seed(1002, rank))
    out[rank] = (red, seeds)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    for r in range(world):
        red, seeds = out[r]
        assert red == [15.0, 3.0]          # max over ranks, element-wise
        assert seeds == [1002, 1003]       # distinct replicas
    import bench

    # two replicas, each 3.88e12 effective FLOP per step, slowest rank 10 ms per step
    assert abs(bench.whole_job_tflops(3.88e12, 2, 10.0) - 776.0) < 1e-6


def test_single_process_needs_no_process_group():
    import bench

    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
