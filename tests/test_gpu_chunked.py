"""GPU parity of chunked prefill against a KV cache (attn_fwd_chunked).

Query row i of sequence b sits at key position q_pos[b] + i and sees the
cache keys below kv_lens[b] ("Implementing attention from scratch", KV
caching).  Cache rows at or past kv_lens hold NaN in every case here: they
must never reach the result.  Cases cover ragged chunks (rows past a
sequence's chunk are padded rows), chunk starts that are not multiples of
the 128-row tile, GQA, bf16 on the tensor cores (D 64 and 128) and the exact
float32 path.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from parity import compare, oracle_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


def _case(B, Hq, Hkv, T, S_max, D, dtype, q_pos, chunk_lens, seed):
    """Random q and caches; cache rows at or past q_pos + chunk_len are NaN."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.randn(B, Hq, T, D, generator=g, device="cuda").to(dt)
    kc = torch.randn(B, Hkv, S_max, D, generator=g, device="cuda").to(dt)
    vc = torch.randn(B, Hkv, S_max, D, generator=g, device="cuda").to(dt)
    qp = torch.tensor(q_pos, dtype=torch.int32, device="cuda")
    kl = torch.tensor([p + c for p, c in zip(q_pos, chunk_lens)], dtype=torch.int32,
                      device="cuda")
    for b in range(B):
        kc[b, :, int(kl[b]):] = float("nan")
        vc[b, :, int(kl[b]):] = float("nan")
    return q, kc, vc, qp, kl


CASES = [
    # (B, Hq, Hkv, T, S_max, D, dtype, q_pos, chunk_lens, causal)
    (2, 4, 2, 128, 512, 128, "bf16", [0, 300], [128, 77], True),
    (3, 2, 2, 300, 1100, 64, "bf16", [5, 700, 0], [300, 1, 129], True),
    (2, 8, 2, 257, 900, 128, "bf16", [513, 129], [257, 200], True),
    (2, 4, 4, 64, 700, 128, "bf16", [611, 0], [64, 64], False),
    (1, 2, 1, 200, 333, 64, "bf16", [133], [200], True),
    (2, 4, 2, 100, 400, 64, "f32", [37, 250], [100, 63], True),
    (2, 2, 2, 40, 200, 32, "f32", [160, 0], [40, 17], False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c[6]}-D{c[5]}-T{c[3]}-c{int(c[9])}")
def test_chunked_prefill(E, case):
    B, Hq, Hkv, T, S_max, D, dtype, q_pos, chunk_lens, causal = case
    q, kc, vc, qp, kl = _case(B, Hq, Hkv, T, S_max, D, dtype, q_pos, chunk_lens, seed=11)
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd_chunked(q, kc, vc, qp, kl, causal=causal, scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle_fwd(q, kc, vc, causal, kl, scale, q_pos=qp)
    compare(o, lse, ro, rl, q.dtype, f"chunked {case}")
    assert E.attn_device_error(clear=True) == 0


@pytest.mark.parametrize("D", [64, 128])
def test_chunks_compose_to_full_forward(E, D):
    """One 700-token sequence per batch entry, prefilled in chunks of
    different sizes against a growing cache, gives the rows of one causal
    attn_fwd over the whole sequence."""
    B, Hq, Hkv, N = 2, 4, 2, 700
    g = torch.Generator(device="cuda").manual_seed(21)
    Q = torch.randn(B, Hq, N, D, generator=g, device="cuda").to(torch.bfloat16)
    K = torch.randn(B, Hkv, N, D, generator=g, device="cuda").to(torch.bfloat16)
    V = torch.randn(B, Hkv, N, D, generator=g, device="cuda").to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    full_o, full_l = E.attn_fwd(Q, K, V, causal=True, scale=scale)
    kc = torch.full((B, Hkv, N + 64, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = kc.clone()
    out = torch.zeros_like(Q)
    lse = torch.zeros(B, Hq, N, device="cuda")
    bounds = [0, 1, 130, 131, 400, 401, 700]
    for c0, c1 in zip(bounds[:-1], bounds[1:]):
        kc[:, :, c0:c1] = K[:, :, c0:c1]
        vc[:, :, c0:c1] = V[:, :, c0:c1]
        qp = torch.full((B,), c0, dtype=torch.int32, device="cuda")
        kl = torch.full((B,), c1, dtype=torch.int32, device="cuda")
        o, l = E.attn_fwd_chunked(Q[:, :, c0:c1].contiguous(), kc, vc, qp, kl, scale=scale)
        out[:, :, c0:c1] = o
        lse[:, :, c0:c1] = l
    torch.cuda.synchronize()
    ro, rl = oracle_fwd(Q, K, V, True, None, scale)
    compare(out, lse, ro, rl, torch.bfloat16, "chunks vs oracle")
    # and against the GPU's own full pass: the same rows, within rounding
    d = (out.float() - full_o.float()).abs()
    assert d.max().item() <= 1.5e-2 and d.mean().item() <= 2e-3
    assert (lse - full_l).abs().max().item() <= 2e-3
    assert E.attn_device_error(clear=True) == 0


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 64), ("f32", 64)])
def test_padded_keys_may_hold_nan(E, dtype, D):
    """attn_fwd with key_lens: K/V rows at or past the valid length are NaN
    and must not reach the result (their weight is 0, but 0 * NaN is NaN)."""
    B, H, T = 3, 4, 300
    g = torch.Generator(device="cuda").manual_seed(31)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.randn(B, H, T, D, generator=g, device="cuda").to(dt)
    k = torch.randn(B, H, T, D, generator=g, device="cuda").to(dt)
    v = torch.randn(B, H, T, D, generator=g, device="cuda").to(dt)
    kl = torch.tensor([300, 141, 77], dtype=torch.int32, device="cuda")
    for b in range(B):
        k[b, :, int(kl[b]):] = float("nan")
        v[b, :, int(kl[b]):] = float("nan")
    scale = 1.0 / math.sqrt(D)
    for causal in (True, False):
        o, lse = E.attn_fwd(q, k, v, causal=causal, key_lens=kl, scale=scale)
        torch.cuda.synchronize()
        ro, rl = oracle_fwd(q, k, v, causal, kl, scale)
        compare(o, lse, ro, rl, dt, f"nan padding {dtype} D{D} causal={causal}")
    assert E.attn_device_error(clear=True) == 0


def test_chunked_rejects_missing_arrays(E):
    import ctypes
    lib = E.load()
    rc = lib.attn_fwd_chunked(None, None, None, None, None, None, None, 1, 1, 1, 1, 1, 64,
                              E.ATTN_BF16, 1, ctypes.c_float(0.125), None)
    assert rc == E.ATTN_ERR_INVALID_ARG
