"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1), each with its own shard of
requests (weak scaling, no data-path collective); the only exchange is the max of the step times
over ranks, and the whole-job throughput counts every rank's tokens within that time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from workload import CONFIGS, make_layout


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


def _shard_rank(rank, world, port, names, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://")
    try:
        w, r, _ = bench._dist()
        mine = {}
        for name in names:
            reqs = make_layout(CONFIGS[name], shard=r)     # what bench.py builds on rank r
            mine[name] = (sum(q.n_cached + q.n_query for q in reqs), sum(q.n_sel for q in reqs),
                          [(s.phys_first_page, s.pos0) for q in reqs for s in q.spans])
        gathered = [None] * w
        dist.all_gather_object(gathered, mine)
        out[rank] = gathered
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_hold_different_shards_of_the_same_size():
    """Under weak scaling each rank draws its own requests: equal token and recompute counts (so
    the job throughput is world x one rank's tokens), different span placements; rank 0's shard
    is the single-GPU workload."""
    world, names = 2, ["concurrent_reuse", "batch70b"]
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_shard_rank, args=(world, _free_port(), names, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]                      # every rank saw the same gathered shards
    shards = res[0]
    for name in names:
        (t0, s0, p0), (t1, s1, p1) = shards[0][name], shards[1][name]
        assert (t0, s0) == (t1, s1) and p0 != p1
        single = make_layout(CONFIGS[name])
        assert p0 == [(s.phys_first_page, s.pos0) for q in single for s in q.spans]
        ms = 3.0
        assert bench._job_throughput(t0, world, ms) == pytest.approx((t0 + t1) / (ms / 1e3))
