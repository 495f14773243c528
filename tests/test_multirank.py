"""The benchmark's multi-rank host logic on CPU with the gloo backend at
world size 2: ranks agree on the slowest rank's time, and the whole-job rate
counts every rank's work (weak scaling, no collective on the data path)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.max_over_ranks(10.0 + 5.0 * rank)  # rank 1 is the slow one
        out[rank] = (ms, bench.job_rate(7.7e12, world, ms))
    finally:
        dist.destroy_process_group()


def test_gloo_world_size_two_max_time_and_job_rate():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == pytest.approx(15.0)
    assert out[0][1] == pytest.approx(2 * 7.7e12 / 15e-3)


def test_single_process_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_rate(1e12, 1, 1.0) == pytest.approx(1e15)
