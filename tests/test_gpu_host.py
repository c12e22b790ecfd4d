"""GPU tests of attn_fwd_host: the prefill on host buffers, copied in,
computed and copied out in pipelined stages over three streams.

The computation is attn_fwd's ("Implementing attention from scratch", Core
ideas: Shapes first, Masks, Stable softmax): the same kernels run on each
stage's (sequence, KV head) range, and a row's arithmetic does not depend on
which rows share a launch, so O and LSE must equal attn_fwd's bit for bit.
Cases cover one stage and several (ragged last stage; stages of whole
sequences and of KV heads inside one sequence), GQA, key padding, fp16 and
fp32, LSE omitted, copies on the compute stream, pageable host memory, and
one comparison with the float64 oracle.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from parity import TOL, compare, oracle_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


def _inputs(B, Hq, Hkv, T, S, D, dtype, seed, lens=None):
    g = torch.Generator(device="cuda").manual_seed(seed)
    q = torch.randn(B, Hq, T, D, generator=g, device="cuda").to(dtype)
    k = torch.randn(B, Hkv, S, D, generator=g, device="cuda").to(dtype)
    v = torch.randn(B, Hkv, S, D, generator=g, device="cuda").to(dtype)
    kl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    return q, k, v, kl


def _stages(E, B, Hkv, in_bytes):
    """The stage count the library picks (about 32 MiB of inputs each)."""
    units = B * Hkv
    want = min(16, max(1, -(-in_bytes // (32 << 20))))
    per = -(-units // want)
    if per >= Hkv:
        nb = -(-per // Hkv)
        return -(-B // nb)
    return B * -(-Hkv // per)


CASES = [
    # (dtype, B, Hq, Hkv, T, S, D, causal, lens, pinned, side_streams, lse)
    (torch.bfloat16, 3, 8, 2, 300, 400, 128, True, [400, 17, 250], True, True, True),
    (torch.bfloat16, 1, 16, 16, 8192, 8192, 128, True, None, True, True, True),      # 3 stages of heads
    (torch.bfloat16, 8, 4, 4, 2048, 2048, 128, True,
     [2048, 1500, 2047, 1, 777, 2048, 1024, 0], True, True, True),                   # stages of sequences
    (torch.bfloat16, 2, 32, 8, 1024, 3072, 64, False, [3072, 2000], True, True, False),
    (torch.bfloat16, 1, 32, 8, 8192, 8192, 128, True, [8000], True, True, True),      # GQA, 3 stages of KV heads
    (torch.bfloat16, 2, 16, 16, 4096, 4096, 128, True, [4096, 3000], True, True, True),  # 2 stages per sequence
    (torch.float16, 2, 8, 8, 2000, 2000, 128, True, [2000, 1999], True, False, True),  # copies on the compute stream
    (torch.float32, 2, 4, 2, 96, 160, 64, True, [160, 90], False, True, True),        # pageable host memory
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_host_equals_device_call(E, case):
    dtype, B, Hq, Hkv, T, S, D, causal, lens, pinned, side, want_lse = case
    q, k, v, kl = _inputs(B, Hq, Hkv, T, S, D, dtype, seed=B * 1000 + T)
    scale = 1.0 / math.sqrt(D)
    o_dev, lse_dev = E.attn_fwd(q, k, v, causal=causal, key_lens=kl, scale=scale)
    hq, hk, hv = (t.cpu() for t in (q, k, v))
    hkl = None if kl is None else kl.cpu()
    if pinned:
        hq, hk, hv = hq.pin_memory(), hk.pin_memory(), hv.pin_memory()
    o_h = torch.full(q.shape, float("nan"), dtype=dtype, pin_memory=pinned)
    lse_h = torch.full((B, Hq, T), float("nan"), pin_memory=pinned) if want_lse else None
    cin = torch.cuda.Stream() if side else None
    cout = torch.cuda.Stream() if side else None
    before = E.attn_kernel_launches()
    E.attn_fwd_host(hq, hk, hv, o=o_h, lse=lse_h, causal=causal, key_lens=hkl, scale=scale,
                    return_lse=want_lse, copy_in=cin, copy_out=cout)
    torch.cuda.current_stream().synchronize()
    es = q.element_size()
    a = lambda x: -(-x // 256) * 256
    in_bytes = a(B * Hq * T * D * es) + 2 * a(B * Hkv * S * D * es)
    assert E.attn_kernel_launches() - before == _stages(E, B, Hkv, in_bytes)
    iv = torch.int32 if dtype == torch.float32 else torch.int16
    assert torch.equal(o_h.view(iv), o_dev.cpu().view(iv))
    if want_lse:
        assert torch.equal(lse_h.view(torch.int32), lse_dev.cpu().view(torch.int32))


def test_host_matches_oracle(E):
    B, Hq, Hkv, T, S, D = 2, 4, 2, 200, 300, 128
    q, k, v, kl = _inputs(B, Hq, Hkv, T, S, D, torch.bfloat16, seed=7, lens=[300, 120])
    scale = 1.0 / math.sqrt(D)
    o_h, lse_h = E.attn_fwd_host(q.cpu().pin_memory(), k.cpu().pin_memory(),
                                 v.cpu().pin_memory(), causal=True, key_lens=kl.cpu(),
                                 scale=scale, copy_in=torch.cuda.Stream(),
                                 copy_out=torch.cuda.Stream())
    torch.cuda.current_stream().synchronize()
    o_ref, lse_ref = oracle_fwd(q, k, v, True, kl, scale)
    compare(o_h, lse_h, o_ref, lse_ref, torch.bfloat16, what="attn_fwd_host")


def test_host_orders_after_and_before_stream_work(E):
    """Inputs written on the compute stream right before the call are the ones
    copied in, and work enqueued after the call sees the copied-out results."""
    B, Hq, Hkv, T, S, D = 1, 16, 16, 4096, 4096, 128   # two stages
    q, k, v, _ = _inputs(B, Hq, Hkv, T, S, D, torch.bfloat16, seed=11)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    o_h = torch.zeros(q.shape, dtype=torch.bfloat16, pin_memory=True)
    st = torch.cuda.current_stream()
    src = torch.empty(B, Hq, T, D, dtype=torch.bfloat16, device="cuda")
    # a device-side producer on the compute stream: its host copy is the q input
    torch.cuda._sleep(20_000_000)          # keeps the stream busy when the call is enqueued
    src.copy_(q)
    hq2 = torch.empty_like(hq).pin_memory()
    hq2.copy_(src, non_blocking=True)      # on the compute stream
    E.attn_fwd_host(hq2, hk, hv, o=o_h, causal=True, copy_in=torch.cuda.Stream(),
                    copy_out=torch.cuda.Stream())
    back = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    back.copy_(o_h, non_blocking=True)     # after the call on the compute stream
    st.synchronize()
    o_dev, _ = E.attn_fwd(q, k, v, causal=True)
    assert torch.equal(back.view(torch.int16), o_dev.view(torch.int16))


def test_host_call_captures_in_a_graph(E):
    """The call forks to its copy streams and joins back with events, so it
    can be captured in a CUDA graph; replays recompute from the host inputs."""
    B, Hq, Hkv, T, S, D = 1, 16, 16, 4096, 4096, 128   # two stages
    q, k, v, _ = _inputs(B, Hq, Hkv, T, S, D, torch.bfloat16, seed=13)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    o_h = torch.zeros(q.shape, dtype=torch.bfloat16, pin_memory=True)
    lse_h = torch.zeros((B, Hq, T), pin_memory=True)
    ws = torch.empty(E.attn_fwd_host_workspace_size(B, Hq, Hkv, T, S, D, torch.bfloat16),
                     dtype=torch.uint8, device="cuda")
    cin, cout = torch.cuda.Stream(), torch.cuda.Stream()
    E.attn_fwd_host(hq, hk, hv, o=o_h, lse=lse_h, causal=True, workspace=ws, copy_in=cin,
                    copy_out=cout)     # warm (tensor maps, kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        E.attn_fwd_host(hq, hk, hv, o=o_h, lse=lse_h, causal=True, workspace=ws,
                        copy_in=cin, copy_out=cout)
    o_h.zero_()
    lse_h.zero_()
    g.replay()
    torch.cuda.synchronize()
    o_dev, lse_dev = E.attn_fwd(q, k, v, causal=True)
    assert torch.equal(o_h.view(torch.int16), o_dev.cpu().view(torch.int16))
    assert torch.equal(lse_h.view(torch.int32), lse_dev.cpu().view(torch.int32))
    # new host inputs, same graph: the replay reads them
    hq.copy_(torch.flip(hq, dims=[2]))
    g.replay()
    torch.cuda.synchronize()
    o_dev2, _ = E.attn_fwd(hq.cuda(), k, v, causal=True)
    assert torch.equal(o_h.view(torch.int16), o_dev2.cpu().view(torch.int16))
