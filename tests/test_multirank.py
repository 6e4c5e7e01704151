"""The benchmark's multi-rank path (independent replicas, slowest rank sets the
job time) on CPU with world size 2 over gloo."""
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


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    mine = [1.0 + rank, 5.0 - rank, 2.5]  # per-rank timings (ms)
    got = bench.reduce_max_over_ranks(mine, dist, torch.device("cpu"))
    dist.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert out[0] == out[1] == [2.0, 5.0, 2.5]


def test_job_throughput_counts_every_rank():
    import bench

    # two replicas, each 1e12 flops in 1 ms -> 2e15 flop/s for the job
    assert bench.job_throughput(1e12, 2, 1.0) == pytest.approx(2e15)
    assert bench.job_throughput(5.0, 1, 1000.0) == pytest.approx(5.0)
