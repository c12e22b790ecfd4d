"""Seeded random shapes through every forward entry point and the backward,
compared with the float64 oracle under the parity tolerances of
tests/parity.py (the backward: those of tests/test_gpu_bwd.py).

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


@pytest.mark.parametrize("seed", range(8))
def test_fuzz_backward(E, seed):
    """attn_bwd on seeded random shapes (bf16), with the bound of
    tests/test_gpu_bwd.py: 2 u A elementwise, 1e-2 normwise."""
    import oracle
    from test_gpu_bwd import check_grad
    from workloads import to_numpy_exact
    rng = np.random.default_rng(5000 + seed)
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.integers(1, 3))
    Hq = Hkv * int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 3))
    T = int(rng.integers(1, 321))
    S = int(rng.integers(1, 361))
    causal = bool(rng.integers(0, 2))
    kl = torch.from_numpy(rng.integers(0, S + 1, size=B).astype(np.int32)).cuda()
    qp = None
    if rng.integers(0, 2):
        qp = torch.from_numpy(np.array([int(rng.integers(-T, S + 1)) for _ in range(B)],
                                       dtype=np.int32)).cuda()
    q, k, v = _tensors(B, Hq, Hkv, T, S, D, torch.bfloat16, seed)
    g = torch.Generator(device="cuda").manual_seed(7000 + seed)
    dout = torch.randn(B, Hq, T, D, generator=g, device="cuda").to(torch.bfloat16)
    scale = 1.0 / math.sqrt(D)
    if qp is None:
        o, lse = E.attn_fwd(q, k, v, causal=causal, key_lens=kl, scale=scale)
    else:
        o, lse = E.attn_fwd_chunked(q, k, v, qp, kl, causal=causal, scale=scale)
    dq, dk, dv = E.attn_bwd(q, k, v, o, dout, lse, causal=causal, key_lens=kl, q_pos=qp,
                            scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    bits = [to_numpy_exact(t)[0] for t in (q, k, v, dout)]
    kw = dict(causal=causal, key_lens=kl.cpu().numpy(), scale=scale, bf16=True,
              q_pos=None if qp is None else qp.cpu().numpy())
    rq, rk, rv, _, rl = oracle.attn_bwd_np(*bits, **kw)
    aq, ak, av = oracle.attn_bwd_magnitudes_np(*bits, **kw)
    check_grad(dq, rq, aq, f"dq seed {seed}")
    check_grad(dk, rk, ak, f"dk seed {seed}")
    check_grad(dv, rv, av, f"dv seed {seed}")
    empty = ~np.isfinite(rl)
    assert np.all(dq.double().cpu().numpy()[empty] == 0)
