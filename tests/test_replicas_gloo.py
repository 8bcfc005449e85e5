"""The benchmark's replica path (one process per GPU, no data-path
collective) on CPU: two gloo ranks, the job time is the slowest rank's and
the throughput counts every rank's units."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local = [10.0 + rank, 3.0 * (world - rank)]
    got = bench.max_over_ranks(local, dist)
    out[rank] = got + [bench.job_throughput(1000.0, world, got[0])]
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    for r in range(world):
        assert out[r][:2] == [11.0, 6.0]
        assert abs(out[r][2] - 2 * 1000.0 / 11e-3) < 1e-6


def test_single_process_keeps_local_values():
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.job_throughput(32768, 1, 8.0) == 32768 / 8e-3
