"""GPU parity of the key-shard prefill (attn_fwd_kv_shard) and the LSE merge
(attn_lse_merge) with the float64 oracle.

"Building a causal self-attention block from scratch in PyTorch", Extending
It: sharding Q/K/V across devices and recombining the results.  Here the
shards live on one GPU: each shard's partial is compared with
oracle.attn_fwd_kv_shard_np, the merge with oracle.lse_merge_np, and a
sequence split into several shards, computed shard by shard and merged,
with the full attention of the C oracle.  Tolerances are those of the
unsharded paths (tests/parity.py): a shard's partial is an attention over
fewer keys, and the merge adds one fp32 rescaling and one output rounding.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import TOL, compare, oracle_fwd
from workloads import to_numpy_exact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


SHARD_CASES = [
    # (dtype, B, Hq, Hkv, T, S_shard, D, causal, k_off, q_pos, key_lens)
    ("bf16", 2, 4, 2, 200, 300, 128, True, 256, [300, 100], [700, 480]),   # straddles the diagonal
    ("bf16", 1, 2, 2, 128, 256, 64, True, 0, [512], [640]),                # every key before the rows
    ("bf16", 2, 2, 1, 96, 160, 128, True, 400, [100, 420], [600, 520]),    # keys after some rows
    ("bf16", 2, 4, 4, 150, 333, 64, False, 128, [0, 0], [300, 2000]),      # non-causal, padding
    ("f16", 2, 4, 2, 130, 257, 128, True, 64, [200, 0], [500, 300]),
    ("f32", 2, 2, 1, 70, 90, 64, True, 40, [60, 10], [160, 75]),
]


def _rand(B, H, n, D, dtype, g):
    x = torch.randn(B, H, n, D, generator=g, device="cuda")
    return x.to({"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype])


@pytest.mark.parametrize("case", SHARD_CASES, ids=lambda c: f"{c[0]}-" + "x".join(map(str, c[1:7]))
                         + f"-c{int(c[7])}-off{c[8]}")
def test_kv_shard_matches_oracle(E, case):
    dtype, B, Hq, Hkv, T, S, D, causal, k_off, qp, kl = case
    g = torch.Generator(device="cuda").manual_seed(71)
    q, k, v = _rand(B, Hq, T, D, dtype, g), _rand(B, Hkv, S, D, dtype, g), _rand(B, Hkv, S, D, dtype, g)
    q_pos = torch.tensor(qp, dtype=torch.int32, device="cuda")
    key_lens = torch.tensor(kl, dtype=torch.int32, device="cuda")
    for b in range(B):   # shard rows at or past the valid length may hold anything
        k[b, :, max(0, kl[b] - k_off):] = float("nan")
        v[b, :, max(0, kl[b] - k_off):] = float("nan")
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd_kv_shard(q, k, v, q_pos, key_lens, k_off, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    qn, bf = to_numpy_exact(q)
    kn, _ = to_numpy_exact(k)
    vn, _ = to_numpy_exact(v)
    ro, rl = oracle.attn_fwd_kv_shard_np(qn, kn, vn, np.array(qp), np.array(kl), k_off,
                                         causal=causal, scale=scale, bf16=bf)
    compare(o, lse, ro, rl, q.dtype, f"shard {case}")


@pytest.mark.parametrize("shape", [(2, 8, 2, 1024, 128, (600, 1024), [0, 300, 700, 1024]),
                                   (4, 16, 16, 2048, 64, (1024, 2048), [0, 512, 1024, 1536, 2048])],
                         ids=["B2-H8-T1024-D128-3shards", "B4-H16-T2048-D64-4shards"])
def test_sharded_prefill_on_one_gpu_equals_full(E, shape):
    """A causal self-attention prefill with key padding, its keys split into
    shards, each shard's partial computed on its own, merged: the full
    attention (the second shape launches well over 2 x 148 work items per
    shard)."""
    B, Hq, Hkv, T, D, lens, cuts = shape
    x = workloads.prefill_inputs(B, Hq, Hkv, T, T, D, "bf16", seed=72, device="cuda", lens=lens)
    scale = 1.0 / math.sqrt(D)
    q_pos = torch.zeros(B, dtype=torch.int32, device="cuda")      # self-attention: rows at 0..T-1
    n = len(cuts) - 1
    o_parts = torch.empty((n, B, Hq, T, D), dtype=x["q"].dtype, device="cuda")
    lse_parts = torch.empty((n, B, Hq, T), dtype=torch.float32, device="cuda")
    for s, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        E.attn_fwd_kv_shard(x["q"], x["k"][:, :, a:b].contiguous(), x["v"][:, :, a:b].contiguous(),
                            q_pos, x["key_lens"], a, o=o_parts[s], lse=lse_parts[s], causal=True,
                            scale=scale)
    o, lse = E.attn_lse_merge(o_parts, lse_parts)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], True, x["key_lens"], scale)
    compare(o, lse, ro, rl, torch.bfloat16, f"{n} shards merged")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_lse_merge_matches_oracle(E, dtype):
    N, B, Hq, T, D = 4, 2, 3, 37, 128 if dtype != "f32" else 64
    g = torch.Generator(device="cuda").manual_seed(73)
    o_parts = _rand(N, B * Hq, T, D, dtype, g).reshape(N, B, Hq, T, D)
    lse_parts = (torch.randn(N, B, Hq, T, generator=g, device="cuda") * 4 + 300.0)
    # some partials saw no key: -inf, anything in their O (NaN here)
    mask = torch.rand(N, B, Hq, T, generator=g, device="cuda") < 0.3
    lse_parts[mask] = float("-inf")
    o_parts[mask] = float("nan")
    lse_parts[:, 0, 0, 5] = float("-inf")                      # a row no partial saw
    o, lse = E.attn_lse_merge(o_parts, lse_parts)
    torch.cuda.synchronize()
    on, _ = to_numpy_exact(o_parts)
    if dtype == "bf16":
        on = oracle.bf16_bits_to_f64(on)
    ro, rl = oracle.lse_merge_np(on.astype(np.float64), lse_parts.double().cpu().numpy())
    fin = np.isfinite(rl)
    got = o.double().cpu().numpy()
    assert np.all(got[~fin] == 0) and torch.all(torch.isneginf(lse.cpu()[torch.from_numpy(~fin)]))
    # fp32 arithmetic, then one rounding of the output to its type
    rel = {"bf16": 2.0 ** -8, "f16": 2.0 ** -10, "f32": 2.0 ** -21}[dtype]
    err = np.abs(got - ro)[fin]
    assert np.all(err <= rel * np.abs(ro[fin]) + 1e-6), err.max()
    assert np.abs(lse.double().cpu().numpy()[fin] - rl[fin]).max() <= 1e-4


def test_shard_rejects_bad_arguments(E):
    x = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    qp = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(E.AttnError) as ex:
        E.attn_fwd_kv_shard(x, x, x, qp, qp, -1)     # negative key offset
    assert ex.value.status == E.ATTN_ERR_INVALID_ARG
    y = torch.zeros(1, 1, 128, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(E.AttnError) as ex:
        E.attn_fwd_kv_shard(y, y, y, qp, qp, 0)      # D = 96 unsupported
    assert ex.value.status == E.ATTN_ERR_UNSUPPORTED
    assert TOL  # the shared tolerances are the ones used above


@pytest.mark.timeout(600)
def test_ring_attention_default_kernels_one_rank(E, tmp_path):
    """ring.ring_attention with its default per-shard compute and merge (this
    library's kernels) in a one-rank NCCL group: one shard holding every key,
    merged alone, equals the oracle's attention.  (Several ranks need several
    GPUs; the exchange order is tested on the CPU with gloo.)"""
    import torch.distributed as dist
    from exact_tiled_attention_49_b300.ring import ring_attention
    store = dist.FileStore(str(tmp_path / "store"), 1)
    dist.init_process_group("nccl", store=store, rank=0, world_size=1,
                            device_id=torch.device("cuda", 0))
    try:
        B, Hq, Hkv, T, S, D = 2, 4, 2, 200, 500, 128
        g = torch.Generator(device="cuda").manual_seed(77)
        q = _rand(B, Hq, T, D, "bf16", g)
        k = _rand(B, Hkv, S, D, "bf16", g)
        v = _rand(B, Hkv, S, D, "bf16", g)
        lens = torch.tensor([500, 333], dtype=torch.int32, device="cuda")
        q_pos = lens - T   # bottom-right: each sequence's queries end at its last key
        scale = 1.0 / math.sqrt(D)
        o, lse = ring_attention(q, k, v, q_pos, lens, [0], causal=True, scale=scale)
        torch.cuda.synchronize()
        o_ref, lse_ref = oracle_fwd(q, k, v, True, lens, scale, q_pos=q_pos)
        compare(o, lse, o_ref, lse_ref, torch.bfloat16, what="ring_attention, one rank")
    finally:
        dist.destroy_process_group()
