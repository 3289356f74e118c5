"""The multi-process plumbing of bench.py on CPU: two gloo ranks, the barrier around the timed
region, the max over ranks of the elapsed time and the whole-job value (weak scaling)."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    bench.dist_init(w, "gloo")
    bench.barrier(w)
    # each rank reports a different elapsed time; every rank sees the slowest
    t = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    v = bench.job_value(w, rows_per_step=289, steps=4, ms_total_max=t)
    bench.barrier(w)
    out[rank] = (t, v)
    torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time_and_the_job_value():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    t0, v0 = out[0]
    t1, v1 = out[1]
    assert t0 == t1 == 15.0
    assert v0 == v1 == pytest.approx(2 * 289 * 4 / 0.015)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.job_value(1, 100, 10, 2.0) == pytest.approx(100 * 10 / 0.002)
