"""GPU tests of attn_decode_append: the new token's K/V rows written into the
caches by the decode's split kernel, in the same launch that reads them.

"Implementing attention from scratch", KV caching: the step appends the new
token at the cache length and attends over every cached row.  The fused call
must give what the two-call form gives (kv_cache_append at kv_lens - 1, then
attn_decode) bit for bit, outputs and cache contents alike: the decode reads
the same values and does the same arithmetic.  One case is also compared
with the float64 oracle (append, then the definition).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from parity import compare, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


CASES = [
    # (dtype, B, Hq, Hkv, S_max, D, kv_lens)
    (torch.bfloat16, 5, 32, 8, 700, 128, [1, 32, 33, 700, 0]),       # sub-tile edges, empty
    (torch.bfloat16, 3, 8, 8, 300, 64, [299, 64, 17]),
    (torch.float16, 4, 16, 1, 1000, 128, [1000, 513, 2, 999]),       # G = 16
    (torch.float32, 3, 8, 2, 600, 64, [600, 257, 256]),              # the fp32 split kernel
    (torch.float32, 2, 4, 4, 300, 128, [1, 0]),
    (torch.bfloat16, 64, 32, 8, 8193, 128, None),                   # the GQA decode workload's shape
]


def _case(dtype, B, Hq, Hkv, S_max, D, lens, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(B, Hq, D, generator=g, device="cuda").to(dtype)
    kc = torch.randn(B, Hkv, S_max, D, generator=g, device="cuda").to(dtype)
    vc = torch.randn(B, Hkv, S_max, D, generator=g, device="cuda").to(dtype)
    kn = torch.randn(B, Hkv, D, generator=g, device="cuda").to(dtype)
    vn = torch.randn(B, Hkv, D, generator=g, device="cuda").to(dtype)
    if lens is None:
        lens = np.random.default_rng(seed).integers(1025, 8194, size=B)
    kv = torch.tensor(np.asarray(lens, dtype=np.int32), device="cuda")
    return q, kc, vc, kn, vn, kv


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_fused_append_equals_two_calls(E, case):
    dtype, B, Hq, Hkv, S_max, D, lens = case
    q, kc, vc, kn, vn, kv = _case(dtype, B, Hq, Hkv, S_max, D, lens, seed=B + S_max)
    scale = 1.0 / math.sqrt(D)
    kc2, vc2 = kc.clone(), vc.clone()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.kv_cache_append(kc2, vc2, kn, vn, kv - 1, dev_status=status)   # kv_lens 0: nothing written
    o_ref, lse_ref = E.attn_decode(q, kc2, vc2, kv, scale=scale)
    before = E.attn_kernel_launches()
    o, lse = E.attn_decode_append(q, kc, vc, kn, vn, kv, scale=scale)
    torch.cuda.synchronize()
    assert E.attn_kernel_launches() - before == 2          # split + merge, no append launch
    iv = torch.int32 if dtype == torch.float32 else torch.int16
    assert torch.equal(kc.view(iv), kc2.view(iv))
    assert torch.equal(vc.view(iv), vc2.view(iv))
    assert torch.equal(o.view(iv), o_ref.view(iv))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))


def test_fused_append_clamps_lengths_past_the_cache(E):
    """kv_lens beyond S_max is clamped to S_max as in attn_decode: the new
    token then lands in the cache's last row."""
    B, Hq, Hkv, S_max, D = 3, 8, 2, 200, 128
    q, kc, vc, kn, vn, kv = _case(torch.bfloat16, B, Hq, Hkv, S_max, D, [205, 200, 1], seed=21)
    scale = 1.0 / math.sqrt(D)
    kc2, vc2 = kc.clone(), vc.clone()
    E.kv_cache_append(kc2, vc2, kn, vn, torch.clamp(kv, max=S_max) - 1)
    o_ref, lse_ref = E.attn_decode(q, kc2, vc2, kv, scale=scale)
    o, lse = E.attn_decode_append(q, kc, vc, kn, vn, kv, scale=scale)
    torch.cuda.synchronize()
    assert torch.equal(kc.view(torch.int16), kc2.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc2.view(torch.int16))
    assert torch.equal(o.view(torch.int16), o_ref.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_ref.view(torch.int32))


def test_fused_append_matches_oracle(E):
    q, kc, vc, kn, vn, kv = _case(torch.bfloat16, 6, 16, 4, 900, 128,
                                  [900, 1, 0, 257, 256, 640], seed=3)
    scale = 1.0 / math.sqrt(128)
    # the oracle's cache: the new rows written at kv_lens - 1 on the host
    kc_h, vc_h = kc.clone(), vc.clone()
    for b, L in enumerate(kv.tolist()):
        if L > 0:
            kc_h[b, :, L - 1] = kn[b]
            vc_h[b, :, L - 1] = vn[b]
    o, lse = E.attn_decode_append(q, kc, vc, kn, vn, kv, scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_decode(q, kc_h, vc_h, kv, scale)
    compare(o, lse, o_ref, lse_ref, torch.bfloat16, what="attn_decode_append")
    assert torch.equal(kc.view(torch.int16), kc_h.view(torch.int16))
    assert torch.equal(vc.view(torch.int16), vc_h.view(torch.int16))
