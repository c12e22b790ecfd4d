"""GPU parity on the paths the kernels take at full size, for every input type.

The persistent prefill deals its work items (pairs of 128-row query tiles)
over the SMs; only a launch with more items than SMs exercises the walk to a
CTA's next item, the next item's early start during the causal diagonal step,
the reuse of the Q buffers and the K/V ring carried across items.  The decode
kernel likewise only reaches its later work when the cache holds more work
than its workers take at once.  "Implementing attention from scratch",
Testing against a reference and Common misconceptions: one small random
input proves little; lengths, padding, dtypes and gradients need their own
checks.  Each case below launches well over 2 x 148 work items:

* bf16, D = 64: B=8 Hq=16 Hkv=4 T=S=2048, causal + key padding (1152
  items), every row against the float64 oracle;
* fp16 at the padded-batch shape (B=8 H=16 T=S=4096 D=128, causal + key
  padding; 2176 items) and fp16 D = 64 (B=4 H=16 T=S=2048): sampled rows,
  every padded row exactly 0 / -inf;
* E4M3 at the padded-batch shape and at the long-context shape (B=1 H=16
  T=S=32768): sampled rows within the derived E4M3 bound;
* bf16 D = 64 decode with 32 sequences x 8 KV heads of up to 4096 cached
  keys: every output against the oracle;
* the backward on one sequence of the padded batch (all 16 heads, T=S=4096,
  causal + padding), every gradient element against the float64 oracle;
* chunked prefill against ragged caches with 640 work items (sampled rows,
  every padded row past each chunk exactly 0 / -inf);
* decode with group sizes 16, 1 (fp16) and 8 over thousands of cached keys,
  every output against the oracle; the exact fp32 prefill over several
  hundred blocks.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import (assert_padded_rows_zero, compare, gather_rows, oracle_decode, oracle_fwd,
                    sample_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


def _items(B, Hq, T, padded):
    """Work items of the persistent prefill (pairs of 128-row tiles)."""
    span = T + 128 if padded else T + (128 if ((T + 127) // 128) % 2 else 0)
    return (span + 255) // 256 * B * Hq


def test_bf16_d64_many_items_full(E):
    B, Hq, Hkv, T, S, D = 8, 16, 4, 2048, 2048, 64
    assert _items(B, Hq, T, True) > 2 * 148
    x = workloads.prefill_inputs(B, Hq, Hkv, T, S, D, "bf16", seed=61, device="cuda",
                                 lens=(1024, 2048))
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd(x["q"], x["k"], x["v"], causal=True, key_lens=x["key_lens"],
                        scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], True, x["key_lens"], scale)
    compare(o, lse, ro, rl, torch.bfloat16, "bf16 D64 B8 H16 T2048 causal+pad")
    assert_padded_rows_zero(o, lse, x["key_lens"].cpu().numpy(), S)


@pytest.mark.parametrize("shape", [(8, 16, 16, 4096, 128, (2048, 4096)),
                                   (4, 16, 16, 2048, 64, None)],
                         ids=["padded-batch-D128", "B4-H16-T2048-D64"])
def test_f16_many_items_sampled(E, shape):
    B, Hq, Hkv, T, D, lens = shape
    S = T
    assert _items(B, Hq, T, lens is not None) > 2 * 148
    x = workloads.prefill_inputs(B, Hq, Hkv, T, S, D, "f16", seed=62, device="cuda", lens=lens)
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd(x["q"], x["k"], x["v"], causal=True, key_lens=x["key_lens"],
                        scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    kl = None if lens is None else x["key_lens"].cpu().numpy()
    rows = sample_rows(B, Hq, T, S, kl, per_head=24, seed=62)
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], True, x["key_lens"], scale, rows=rows)
    og, lg = gather_rows(o, lse, rows, D)
    compare(og, lg, ro, rl, torch.float16, f"f16 {shape} (sampled rows)")
    if kl is not None:
        assert_padded_rows_zero(o, lse, kl, S)


def _fp8(x: torch.Tensor, descale: float) -> torch.Tensor:
    return (x / descale).to(torch.float8_e4m3fn)


def _n_visible(rows, Hq, T, S, lens, causal):
    i = rows % T
    b = rows // (Hq * T)
    L = np.full(i.shape, S) if lens is None else np.asarray(lens)[b]
    pos = i + (S - T)
    lim = np.minimum(L, pos + 1) if causal else L
    return np.where(pos < L, np.maximum(lim, 0), 0).astype(np.float64)


@pytest.mark.parametrize("shape", [(8, 16, 4096, (2048, 4096), 16),
                                   (1, 16, 32768, None, 48)],
                         ids=["padded-batch", "long-context"])
def test_fp8_many_items_sampled(E, shape):
    """E4M3 inputs at the two benchmark shapes, sampled rows within the bound
    derived in tests/test_gpu_fp8.py: per element
    1.25 (2^-4 w.|v| + 2^-17 sum_visible |v| + 2^-9 |o|) + 1e-6, with w.|v|
    the attention of |v| and the sum over the row's visible keys."""
    B, H, T, lens, per_head = shape
    S, D = T, 128
    assert _items(B, H, T, lens is not None) > 2 * 148
    qd, kd, vd = 0.25, 0.5, 0.125
    g = torch.Generator(device="cuda").manual_seed(63)
    q = _fp8(torch.randn(B, H, T, D, generator=g, device="cuda"), qd)
    k = _fp8(torch.randn(B, H, S, D, generator=g, device="cuda"), kd)
    v = _fp8(torch.randn(B, H, S, D, generator=g, device="cuda"), vd)
    kl, lens_np = None, None
    if lens is not None:
        lens_np = workloads.lengths(63, lens[0], lens[1], B)
        kl = torch.from_numpy(lens_np).cuda()
        kb, vb = k.view(torch.uint8), v.view(torch.uint8)
        for b in range(B):   # padded rows may hold anything: E4M3 NaN codes here
            kb[b, :, int(lens_np[b]):] = 0x7F
            vb[b, :, int(lens_np[b]):] = 0x7F
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd_fp8(q, k, v, causal=True, key_lens=kl, scale=scale,
                            q_descale=qd, k_descale=kd, v_descale=vd)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    rows = sample_rows(B, H, T, S, lens_np, per_head=per_head, seed=63)
    qf = oracle.e4m3_bits_to_f64(q.view(torch.uint8).cpu().numpy()) * qd
    kf = oracle.e4m3_bits_to_f64(k.view(torch.uint8).cpu().numpy()) * kd
    vf = oracle.e4m3_bits_to_f64(v.view(torch.uint8).cpu().numpy()) * vd
    ro, rl = oracle.attn_fwd(qf, kf, vf, causal=True, key_lens=lens_np, scale=scale, rows=rows)
    av = np.abs(np.nan_to_num(vf))
    wa, _ = oracle.attn_fwd(qf, kf, av, causal=True, key_lens=lens_np, scale=scale, rows=rows)
    # Q = 0 weighs every visible key equally: the mean of the visible |v| rows
    um, _ = oracle.attn_fwd(np.zeros_like(qf), kf, av, causal=True, key_lens=lens_np,
                            scale=scale, rows=rows)
    usum = um * _n_visible(rows, H, T, S, lens_np, True)[:, None]
    bound = 1.25 * (2.0 ** -4 * wa + 2.0 ** -17 * usum + 2.0 ** -9 * np.abs(ro)) + 1e-6
    og, lg = gather_rows(o, lse, rows, D)
    got = og.double().cpu().numpy()
    gl = lg.double().cpu().numpy()
    valid = np.isfinite(rl)
    assert np.isfinite(got).all()
    err = np.abs(got - ro)
    assert np.all(err[valid] <= bound[valid]), f"max excess {(err - bound)[valid].max():.3g}"
    assert np.all(got[~valid] == 0) and np.all(np.isneginf(gl[~valid]))
    assert np.abs(gl[valid] - rl[valid]).max() <= 2e-3
    if lens_np is not None:
        assert_padded_rows_zero(o, lse, lens_np, S)


def test_bf16_d64_decode_many_items_full(E):
    B, Hq, Hkv, D = 32, 32, 8, 64
    d = workloads.decode_inputs(B, Hq, Hkv, D, 1024, 4096, "bf16", seed=64, device="cuda")
    E.kv_cache_append(d["kcache"], d["vcache"], d["k_new"], d["v_new"], d["cache_len"])
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_decode(d["q"], d["kcache"], d["vcache"], d["kv_len"], scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    # 256-key chunks per (sequence, KV head): far more than the workers
    chunks = int(((d["kv_len"].cpu().numpy() + 255) // 256).sum()) * Hkv
    assert chunks > 8 * 148
    ro, rl = oracle_decode(d["q"], d["kcache"], d["vcache"], d["kv_len"], scale)
    compare(o, lse, ro, rl, torch.bfloat16, "bf16 D64 decode B32 Hq32 Hkv8")


def test_backward_padded_batch_slice(E):
    """One sequence of the padded batch, all 16 heads, T=S=4096, causal with
    its key padding; every element of dQ, dK, dV within the derived bound of
    tests/test_gpu_bwd.py (4 u A elementwise, 1e-2 normwise)."""
    from test_gpu_bwd import check_grad
    from workloads import to_numpy_exact
    w = workloads.WORKLOADS[5]
    L = int(workloads.lengths(5, w.lens[0], w.lens[1], w.B)[0])
    B, H, T, S, D = 1, w.Hq, w.T, w.S, w.D
    g = torch.Generator(device="cuda").manual_seed(65)
    q, k, v, dout = (torch.randn(B, H, n, D, generator=g, device="cuda").to(torch.bfloat16)
                     for n in (T, S, S, T))
    kl = torch.tensor([L], dtype=torch.int32, device="cuda")
    k[:, :, L:] = float("nan")     # rows past the valid length may hold anything
    v[:, :, L:] = float("nan")
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd(q, k, v, causal=True, key_lens=kl, scale=scale)
    dq, dk, dv = E.attn_bwd(q, k, v, o, dout, lse, causal=True, key_lens=kl, scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    bits = [to_numpy_exact(t)[0] for t in (q, k, v, dout)]
    lens = np.array([L], np.int32)
    rq, rk, rv, _, rl = oracle.attn_bwd_np(*bits, causal=True, key_lens=lens, scale=scale,
                                           bf16=True)
    aq, ak, av = oracle.attn_bwd_magnitudes_np(*bits, causal=True, key_lens=lens, scale=scale,
                                               bf16=True)
    check_grad(dq, rq, aq, "dq")
    check_grad(dk, rk, ak, "dk")
    check_grad(dv, rv, av, "dv")
    assert np.all(dq.double().cpu().numpy()[~np.isfinite(rl)] == 0)
    assert torch.all(dk[:, :, L:] == 0) and torch.all(dv[:, :, L:] == 0)


def test_chunked_prefill_many_items_sampled(E):
    """Chunked prefill against caches (ragged cache lengths, ragged chunks)
    with 640 work items: q_pos[b] is the cache length before the chunk,
    kv_lens[b] = q_pos[b] + that sequence's chunk length (<= T); cache rows
    past kv_lens hold NaN."""
    B, Hq, Hkv, T, S_max, D = 8, 16, 4, 1024, 4096, 128
    assert _items(B, Hq, T, True) > 2 * 148
    g = torch.Generator(device="cuda").manual_seed(66)
    q = torch.randn(B, Hq, T, D, generator=g, device="cuda").to(torch.bfloat16)
    kc = torch.randn(B, Hkv, S_max, D, generator=g, device="cuda").to(torch.bfloat16)
    vc = torch.randn(B, Hkv, S_max, D, generator=g, device="cuda").to(torch.bfloat16)
    rng = np.random.default_rng(66)
    qp = rng.integers(0, S_max - T + 1, size=B).astype(np.int32)
    chunk = rng.integers(1, T + 1, size=B).astype(np.int32)
    kl = (qp + chunk).astype(np.int32)
    for b in range(B):
        kc[b, :, int(kl[b]):] = float("nan")
        vc[b, :, int(kl[b]):] = float("nan")
    q_pos = torch.from_numpy(qp).cuda()
    kv_lens = torch.from_numpy(kl).cuda()
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd_chunked(q, kc, vc, q_pos, kv_lens, scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    rows = sample_rows(B, Hq, T, S_max, kl, per_head=16, seed=66, q_off=0)
    # the rows around each sequence's chunk end too
    extra = [(b * Hq + h) * T + i for b in range(B) for h in range(0, Hq, 5)
             for i in (int(chunk[b]) - 1, min(int(chunk[b]), T - 1)) if 0 <= i < T]
    rows = np.unique(np.concatenate([rows, np.array(extra, np.int64)]))
    ro, rl = oracle_fwd(q, kc, vc, True, kv_lens, scale, rows=rows, q_pos=q_pos)
    og, lg = gather_rows(o, lse, rows, D)
    compare(og, lg, ro, rl, torch.bfloat16, "chunked B8 H16 T1024 S_max4096 (sampled rows)")
    for b in range(B):   # rows past each chunk are padded rows
        assert torch.all(o[b, :, int(chunk[b]):] == 0)
        assert torch.all(torch.isneginf(lse[b, :, int(chunk[b]):]))


@pytest.mark.parametrize("cfg", [(16, 32, 2, 128, "bf16"), (24, 8, 8, 64, "f16"),
                                 (16, 64, 8, 64, "bf16")],
                         ids=["G16-D128-bf16", "G1-D64-f16", "G8-D64-bf16"])
def test_decode_group_sizes_at_scale(E, cfg):
    """Decode with group sizes 16, 1 and 8 over thousands of cached keys per
    sequence, every output against the oracle (the balanced split gives each
    warp a span across many streams)."""
    B, Hq, Hkv, D, dtype = cfg
    d = workloads.decode_inputs(B, Hq, Hkv, D, 512, 6000, dtype, seed=67, device="cuda")
    E.kv_cache_append(d["kcache"], d["vcache"], d["k_new"], d["v_new"], d["cache_len"])
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_decode(d["q"], d["kcache"], d["vcache"], d["kv_len"], scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    ro, rl = oracle_decode(d["q"], d["kcache"], d["vcache"], d["kv_len"], scale)
    compare(o, lse, ro, rl, d["q"].dtype, f"decode {cfg}")


@pytest.mark.parametrize("cfg", [(1, 32, 8, 128, 131071, "bf16"), (2, 16, 2, 64, 60000, "f16"),
                                 (3, 8, 1, 128, 20000, "bf16")],
                         ids=["B1-131k-D128", "B2-60k-D64-f16", "B3-20k-G8"])
def test_decode_few_long_streams(E, cfg):
    """Decode of a few long sequences, where every stream is cut into many
    pieces (up to ~111 per stream) and the merge runs one block per head:
    every output against the oracle, through attn_decode_append (the new
    token's rows written by the split kernel)."""
    B, Hq, Hkv, D, n, dtype = cfg
    d = workloads.decode_inputs(B, Hq, Hkv, D, n // 2, n, dtype, seed=71, device="cuda")
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_decode_append(d["q"], d["kcache"], d["vcache"], d["k_new"], d["v_new"],
                                  d["kv_len"], scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    ro, rl = oracle_decode(d["q"], d["kcache"], d["vcache"], d["kv_len"], scale)
    compare(o, lse, ro, rl, d["q"].dtype, f"decode {cfg}")


def test_fp32_prefill_larger(E):
    """The exact fp32 path over several hundred blocks, causal with padding."""
    x = workloads.prefill_inputs(2, 4, 2, 700, 700, 128, "f32", seed=68, device="cuda",
                                 lens=(300, 700))
    scale = 1.0 / math.sqrt(128)
    o, lse = E.attn_fwd(x["q"], x["k"], x["v"], causal=True, key_lens=x["key_lens"], scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], True, x["key_lens"], scale)
    compare(o, lse, ro, rl, torch.float32, "fp32 B2 H4 T700 D128 causal+pad")
