"""Host logic of bench.py's N > 1 mode ("replicas only": each rank runs its
own replica, no collective on the data path), on CPU with two gloo ranks: the
reported time is the slowest rank's, and the job's throughput counts every
replica's work over that time."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ms = [3.0, 5.0][rank]                      # rank 1 is the slow one
    got = bench.max_over_ranks(ms, dist, torch.device("cpu"))
    dist.barrier()
    out[rank] = got
    dist.destroy_process_group()


def test_slowest_rank_sets_the_time():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert dict(out) == {0: 5.0, 1: 5.0}


def test_job_throughput_counts_every_replica():
    import bench

    assert bench.max_over_ranks(7.0, None, None) == 7.0
    one = bench.job_tflops(1, 120.3e9, 0.1)
    assert bench.job_tflops(2, 120.3e9, 0.1) == pytest.approx(2 * one)
    assert one == pytest.approx(1203.0)
