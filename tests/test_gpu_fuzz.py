"""Seeded random shapes through every forward entry point, compared with the
float64 oracle under the parity tolerances of tests/parity.py.

The fixed cases elsewhere pin the paths the kernels take (tile boundaries,
padding, item walks at full size); these draws add shapes no one picked:
ragged T and S, GQA group sizes 1-8, key lengths anywhere in [0, S] (empty
sequences included), query offsets before, inside and after the cache, both
mask settings and every input type.  "Implementing attention from scratch",
Common misconceptions: one random input proves little, so the draws vary
lengths, padding and types.  Sizes stay small enough for the oracle to
compute every row.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from parity import compare, oracle_decode, oracle_fwd

pytestmark = pytest.mark.gpu

DTYPES = [torch.bfloat16, torch.float16, torch.float32]


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


def _draw(seed):
    rng = np.random.default_rng(seed)
    dtype = DTYPES[int(rng.integers(0, 3))]
    D = int(rng.choice([64, 128])) if dtype != torch.float32 else int(rng.integers(1, 257))
    Hkv = int(rng.integers(1, 4))
    G = int(rng.choice([1, 2, 4, 8]))
    B = int(rng.integers(1, 4))
    T = int(rng.integers(1, 600))
    S = int(rng.integers(1, 700))
    causal = bool(rng.integers(0, 2))
    return rng, dtype, B, Hkv * G, Hkv, T, S, D, causal


def _tensors(B, Hq, Hkv, T, S, D, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(B, Hq, T, D, generator=g, device="cuda").to(dtype)
    k = torch.randn(B, Hkv, S, D, generator=g, device="cuda").to(dtype)
    v = torch.randn(B, Hkv, S, D, generator=g, device="cuda").to(dtype)
    return q, k, v


@pytest.mark.parametrize("seed", range(16))
def test_fuzz_fwd(E, seed):
    rng, dtype, B, Hq, Hkv, T, S, D, causal = _draw(1000 + seed)
    q, k, v = _tensors(B, Hq, Hkv, T, S, D, dtype, seed)
    lens = None
    if rng.integers(0, 2):
        lens = rng.integers(0, S + 1, size=B).astype(np.int32)
        lens[rng.integers(0, B)] = S
    kl = None if lens is None else torch.from_numpy(lens).cuda()
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd(q, k, v, causal=causal, key_lens=kl, scale=scale)
    o_ref, lse_ref = oracle_fwd(q, k, v, causal, kl, scale)
    compare(o, lse, o_ref, lse_ref, dtype, what=f"fwd seed {seed}")


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_chunked(E, seed):
    rng, dtype, B, Hq, Hkv, T, S, D, causal = _draw(2000 + seed)
    q, k, v = _tensors(B, Hq, Hkv, T, S, D, dtype, seed)
    kv_lens = rng.integers(0, S + 1, size=B).astype(np.int32)
    # query offsets from before the cache start to past its valid end
    q_pos = np.array([int(rng.integers(-T - 50, int(l) + 50)) for l in kv_lens], dtype=np.int32)
    kl, qp = torch.from_numpy(kv_lens).cuda(), torch.from_numpy(q_pos).cuda()
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd_chunked(q, k, v, qp, kl, causal=causal, scale=scale)
    o_ref, lse_ref = oracle_fwd(q, k, v, causal, kl, scale, q_pos=qp)
    compare(o, lse, o_ref, lse_ref, dtype, what=f"chunked seed {seed}")


@pytest.mark.parametrize("seed", range(12))
def test_fuzz_decode(E, seed):
    rng, dtype, B, Hq, Hkv, _, S, D, _ = _draw(3000 + seed)
    D = int(rng.choice([64, 128]))   # the decode kernels take D in {64, 128} for every type
    B = int(rng.integers(1, 40))
    S_max = int(rng.integers(1, 3000))
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(B, Hq, D, generator=g, device="cuda").to(dtype)
    kc = torch.randn(B, Hkv, S_max, D, generator=g, device="cuda").to(dtype)
    vc = torch.randn(B, Hkv, S_max, D, generator=g, device="cuda").to(dtype)
    kv = rng.integers(0, S_max + 1, size=B).astype(np.int32)
    kl = torch.from_numpy(kv).cuda()
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_decode(q, kc, vc, kl, scale=scale)
    o_ref, lse_ref = oracle_decode(q, kc, vc, kl, scale)
    compare(o, lse, o_ref, lse_ref, dtype, what=f"decode seed {seed}")


@pytest.mark.parametrize("seed", range(6))
def test_fuzz_host(E, seed):
    rng, dtype, B, Hq, Hkv, T, S, D, causal = _draw(4000 + seed)
    q, k, v = _tensors(B, Hq, Hkv, T, S, D, dtype, seed)
    lens = rng.integers(0, S + 1, size=B).astype(np.int32)
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd_host(q.cpu().pin_memory(), k.cpu().pin_memory(), v.cpu().pin_memory(),
                             causal=causal, key_lens=torch.from_numpy(lens), scale=scale,
                             copy_in=torch.cuda.Stream(), copy_out=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    o_ref, lse_ref = oracle_fwd(q, k, v, causal, torch.from_numpy(lens), scale)
    compare(o, lse, o_ref, lse_ref, dtype, what=f"host seed {seed}")
