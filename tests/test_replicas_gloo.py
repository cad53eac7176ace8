"""The multi-GPU mode is replicas only (one independent step per rank, no
data-path collective).  Its host side -- the barrier, the max over ranks of
the step time, the whole-job value and the rank-0-only reference arm -- runs
here as world-size-2 gloo process groups on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    dist = bench.dist_setup(world, "gloo")
    bench.barrier(dist)
    us = bench.allmax(dist, 100.0 + 50.0 * rank, torch.device("cpu"))   # rank 1 is slower
    value = bench.replica_value(us, world)
    bench.barrier(dist)
    ref = bench.run_reference(type("A", (), {"config": "c1", "steps": 1, "warmup": 1})(), rank, world) if rank else None
    dist.destroy_process_group()
    out.put((rank, us, value, ref))


def test_replicas_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slowest rank's time; the job value counts both replicas
    assert [r[1] for r in res] == [150.0, 150.0]
    assert res[0][2] == pytest.approx(2 * 1e6 / 150.0)
    assert res[1][3] == 0          # the reference arm runs on rank 0 only


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_setup(1) is None
    assert bench.allmax(None, 3.5, None) == 3.5
    assert bench.replica_value(100.0, 1) == pytest.approx(1e4)
