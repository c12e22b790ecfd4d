"""The N > 1 host path of bench.py on CPU: two gloo ranks, no GPU.

bench.py runs one independent replica per GPU; the only cross-rank steps are
a barrier around the timed region and the max-over-ranks reduction of its
time.  These run here with the gloo backend, world size 2, on 127.0.0.1.
"""
from __future__ import annotations

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


def _worker(rank: int, ws: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(ws),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench.dist_env()
        bench.barrier(ws)
        mx = bench.reduce_max(1.5 + rank, ws)          # rank 1 is the slower one
        bench.barrier(ws)
        # the reference arm: every rank but 0 returns at once, without work
        ran = None
        if rank != 0:
            class A:
                workload, steps, warmup = 2, 1, 3
            bench.bench_reference(A())
            ran = "returned"
        q.put((rank, got_ws, got_rank, got_local, mx, ran))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    assert [r[1] for r in res] == [2, 2]
    assert [r[2] for r in res] == [0, 1] and [r[3] for r in res] == [0, 1]
    assert all(r[4] == pytest.approx(2.5) for r in res)  # max over ranks on every rank
    assert res[1][5] == "returned"


def test_single_process_helpers_are_identities(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.reduce_max(3.25, 1) == 3.25
    bench.barrier(1)
