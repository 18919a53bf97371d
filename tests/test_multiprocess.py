"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1), each with its own copy of the
workload (weak scaling, no data-path collective); the only exchange is the max of the step times
over ranks, and the whole-job throughput counts every rank's tokens within that time."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://")
    try:
        w, r, local = bench._dist()
        assert (w, r, local) == (world, rank, rank)
        ms = bench._max_over_ranks(times[rank], w, "cpu")
        out[rank] = (ms, bench._job_throughput(1000, w, ms))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(2.0, 3.5), (7.25, 1.0)])
def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_throughput(times):
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    slowest = max(times)
    for rank in range(world):
        ms, tput = res[rank]
        assert ms == slowest
        assert tput == pytest.approx(world * 1000 / (slowest / 1e3))


def test_single_rank_needs_no_process_group():
    assert bench._max_over_ranks(4.0, 1, "cpu") == 4.0
    assert bench._job_throughput(500, 1, 2.0) == pytest.approx(250000.0)
