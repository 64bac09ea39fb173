"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each timing one replica of the
workload, report the slowest rank's time and the whole job's throughput (weak scaling)."""
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


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        assert (w, r, local) == (world, rank, rank)
        ms = bench.max_over_ranks(times[rank], w, torch.device("cpu"))
        dist.barrier()
        out[rank] = ms
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    times = [3.5, 7.25]
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
    assert out[0] == out[1] == max(times)


def test_whole_job_throughput_counts_every_replica():
    # 9.07 TFLOP per replica step, 10 ms per step: 907 TFLOP/s on one rank, twice that on two
    assert bench.job_tflops(1, 9.07e12, 10.0) == pytest.approx(907.0)
    assert bench.job_tflops(2, 9.07e12, 10.0) == pytest.approx(1814.0)
    assert bench.max_over_ranks(4.0, 1, torch.device("cpu")) == 4.0
