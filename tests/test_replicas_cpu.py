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


def test_kernel_hash_follows_code_not_comments():
    """The kernel hash that ties a committed DRAM-traffic figure to the
    sources it was measured on changes with the code and not with comments,
    blank lines or trailing blanks; comment markers inside string literals
    are code."""
    import bench
    src = 'int a = 1;  // one\n/* block\n comment */\nconst char* s = "x//y";\n\n'
    assert bench.code_only(src) == 'int a = 1;\nconst char* s = "x//y";'
    base = {f: "int f() { return 1; }\n" for f in bench.KERNEL_SOURCES}

    def reader(files):
        return lambda name: files[name]

    h0 = bench.kernel_hash(reader(base))
    commented = dict(base)
    commented[bench.KERNEL_SOURCES[0]] = "// a comment\nint f() { return 1; }   /* trailing */\n\n"
    assert bench.kernel_hash(reader(commented)) == h0
    changed = dict(base)
    changed[bench.KERNEL_SOURCES[0]] = "int f() { return 2; }\n"
    assert bench.kernel_hash(reader(changed)) != h0
