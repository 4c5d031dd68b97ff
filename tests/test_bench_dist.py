"""The bench's multi-rank plumbing on CPU: two gloo ranks, the barrier and
the max-over-ranks of the timed interval (the only collectives the bench
uses; there is none on the data path)."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), BENCH_DIST_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import bench
    r, lr, w = bench.dist_setup()
    bench.dist_barrier(w)
    t = bench.dist_max(1.0 + r, w)          # rank r "took" 1 + r seconds
    bench.dist_barrier(w)
    import torch.distributed as dist
    dist.destroy_process_group()
    results.put((r, lr, w, t))


def test_two_gloo_ranks_agree_on_the_slowest_time():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 0, 2, 2.0), (1, 1, 2, 2.0)]


def test_single_process_needs_no_process_group(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench.dist_setup() == (0, 0, 1)
    assert bench.dist_max(3.5, 1) == 3.5
