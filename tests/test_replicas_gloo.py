"""The multi-rank path of the bench (replicas only: every rank runs the whole
layer on its own sequences, no data-path collective): the job's time is the
slowest rank's, and the job's rate counts every rank's steps.  Run as two gloo
ranks on the CPU."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
        q.put((rank, ms, bench.job_rate(1000, ms, world)))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, rate in got:
        assert ms == pytest.approx(15.0)
        assert rate == pytest.approx(2 * 1000 / 0.015)


def test_one_rank_is_its_own_job():
    assert bench.max_over_ranks(7.5, None, "cpu") == 7.5
    assert bench.job_rate(300, 1500.0, 1) == pytest.approx(200.0)
