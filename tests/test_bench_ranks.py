"""The benchmark's multi-rank logic on CPU with two gloo ranks: every rank runs
an independent replica, the reported time is the max over ranks and the rate
counts the units of all ranks.  No GPU and no data-path collective involved."""
import os
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                 # rank 1 is the slow one
        got = bench.max_over_ranks(ms)
        rate = bench.whole_job_rate(512, world, got / 1e3)
        q.put((rank, got, rate, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_rate():
    world, port = 2, 29517
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got, rate, env in res:
        assert got == 15.0
        assert rate == pytest.approx(2 * 512 / 0.015)
        assert env[0] == rank and env[1] == world


def test_single_process_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(100, 1, 0.5) == 200
