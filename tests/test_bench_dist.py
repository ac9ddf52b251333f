"""bench.py's multi-rank plumbing on CPU: world size 2 over gloo (127.0.0.1)."""

from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import bench
    w, r, _ = bench.dist_setup(want_gpu=False)
    bench.barrier()
    worst = bench.max_over_ranks(1.5 + r)  # each rank's own time; the slowest rank wins
    q.put((r, w, worst))
    dist.destroy_process_group()


def test_two_rank_barrier_and_max_over_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert got == [(0, 2, 2.5), (1, 2, 2.5)]


def test_single_process_defaults():
    import bench
    os.environ.pop("WORLD_SIZE", None)
    w, r, _ = bench.dist_setup(want_gpu=False)
    assert (w, r) == (1, 0)
    assert bench.max_over_ranks(3.0) == 3.0
