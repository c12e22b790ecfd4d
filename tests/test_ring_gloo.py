"""The exchange of sequence-parallel attention on CPU: gloo ranks, no GPU.

exact_tiled_attention_49_b300.ring.ring_attention passes key/value shards
round a ring of ranks and merges each rank's partials.  Here two and three
gloo ranks on 127.0.0.1 run it with the per-shard attention and the merge
taken from the float64 oracle, on a causal self-attention with key padding
and GQA whose queries and keys are split evenly over the ranks.  Checked:
at step s rank r computes the shard of rank (r - s) mod N with that shard's
global key offset; every shard reaches every rank once; the merged result
of each rank's query rows is the full attention (C oracle) of those rows.
"""
from __future__ import annotations

import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

B, HQ, HKV, D, T_PER = 2, 4, 2, 8, 12


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _problem(world):
    T = T_PER * world
    r = np.random.default_rng(5)
    q = r.standard_normal((B, HQ, T, D))
    k = r.standard_normal((B, HKV, T, D))
    v = r.standard_normal((B, HKV, T, D))
    lens = np.array([T, T - 7], np.int32)
    return q, k, v, lens


def _worker(rank, world, port, out_q):
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch
    import torch.distributed as dist
    import oracle
    from exact_tiled_attention_49_b300.ring import ring_attention
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, lens = _problem(world)
        rows = slice(rank * T_PER, (rank + 1) * T_PER)
        calls = []

        def shard_fn(q_, k_, v_, q_pos, key_lens, k_off, o, lse, causal, scale):
            calls.append(int(k_off))
            ro, rl = oracle.attn_fwd_kv_shard_np(q_.numpy(), k_.numpy(), v_.numpy(),
                                                 q_pos.numpy(), key_lens.numpy(), k_off,
                                                 causal=causal, scale=scale)
            o.copy_(torch.from_numpy(ro))
            lse.copy_(torch.from_numpy(rl))

        def merge_fn(o_parts, lse_parts):
            return oracle.lse_merge_np(o_parts.numpy(), lse_parts.double().numpy())

        q_pos = torch.full((B,), rank * T_PER, dtype=torch.int32)
        o, lse = ring_attention(torch.from_numpy(q[:, :, rows].copy()),
                                torch.from_numpy(k[:, :, rows].copy()),
                                torch.from_numpy(v[:, :, rows].copy()),
                                q_pos, torch.from_numpy(lens),
                                [w * T_PER for w in range(world)], causal=True,
                                scale=1.0 / np.sqrt(D), shard_fn=shard_fn, merge_fn=merge_fn)
        ref_o, ref_l = oracle.attn_fwd(q, k, v, causal=True, key_lens=lens, nthreads=1)
        out_q.put((rank, calls, float(np.abs(o - ref_o[:, :, rows]).max()),
                   bool(np.array_equal(np.isneginf(lse), np.isneginf(ref_l[:, :, rows]))),
                   float(np.nanmax(np.abs(np.where(np.isfinite(lse), lse, 0)
                                          - np.where(np.isfinite(ref_l[:, :, rows]),
                                                     ref_l[:, :, rows], 0))))))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_ring_exchange_order_and_result(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, calls, err, same_empty, lse_err in res:
        # step s: the shard that started on rank (rank - s) mod N, at its offset
        assert calls == [((rank - s) % world) * T_PER for s in range(world)]
        assert err <= 1e-5, (rank, err)      # partial LSEs travel as float32
        assert same_empty
        assert lse_err <= 1e-5
