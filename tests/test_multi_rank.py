"""The benchmark's multi-rank logic on CPU: two gloo ranks on 127.0.0.1.

Each rank of a torchrun launch runs an independent replica of the workload; only the
timing is collective (barrier before and after, max of the elapsed times over ranks),
and the whole-job tokens/s counts every rank's tokens.  No GPU is used here.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), GQAW_DIST_BACKEND="gloo")
    import bench

    r, w = bench._dist()
    assert (r, w) == (rank, world)
    bench._barrier(w)
    elapsed = 10.0 * (rank + 1)  # rank 1 is the slow one
    slowest = bench._max_over_ranks(elapsed, w)
    out.put((rank, slowest))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(out.get(timeout=5) for _ in range(2))
    assert got == [(0, 20.0), (1, 20.0)]


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench

    monkeypatch.delenv("WORLD_SIZE", raising=False)
    assert bench._dist() == (0, 1)
    assert bench._max_over_ranks(3.5, 1) == 3.5
