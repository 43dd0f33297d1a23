"""Host logic of the multi-GPU benchmark path on CPU: two gloo ranks, each
timing its own replica; the job time is the slowest rank's and the job rate
counts every rank's work."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slower replica
    out[rank] = bench.global_max(local_ms, dist, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1] == 15.0
    # 2 replicas x 1e9 bytes in 15 ms
    assert bench.job_throughput(1e9, world, out[0]) == pytest.approx(2e9 / 0.015)


def test_single_rank_needs_no_process_group():
    assert bench.global_max(3.5) == 3.5
