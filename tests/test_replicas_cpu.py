"""The multi-GPU path of bench.py is N independent replicas (the projection
has no exchange step): every rank streams the same weights, and the job's
time is the slowest rank's. These tests run its host logic as two gloo ranks
on the CPU."""

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 * (rank + 1)          # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        out[rank] = (ms, bench.replica_value(1000, 4, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        procs = [mp.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 20.0
    # 2 replicas x 4 steps x 1000 bytes in 20 ms
    assert res[0][1] == pytest.approx(2 * 4 * 1000 / 0.020 / 1e9)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(7.5, None, "cpu") == 7.5
    assert bench.replica_value(2e9, 10, 1, 1000.0) == pytest.approx(20.0)

