"""The benchmark's multi-rank plumbing on CPU: two gloo ranks, replicas only (no data-path
collective); the reported time is the maximum over ranks."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench

    r, w = bench.init_dist("gloo")
    assert (r, w) == (rank, world)
    bench.barrier(w)
    got = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    out.put((rank, got, bench.dist_env()))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = [out.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert sorted(r for r, _, _ in res) == [0, 1]
    assert all(abs(v - 15.0) < 1e-12 for _, v, _ in res)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
