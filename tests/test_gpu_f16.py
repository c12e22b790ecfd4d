"""GPU parity of the fp16 paths with the float64 oracle.

fp16 inputs use the same kernels as bf16 (tcgen05 kind::f16 MMAs for the
prefill and the backward, mma.sync for the decode), with P and the outputs
rounded to fp16.  Tolerances: the bf16 bounds scaled by the unit roundoff
ratio 2^-11 / 2^-8 times 2 (tests/parity.py), and for the backward the
derived elementwise bound of tests/test_gpu_bwd.py with u = 2^-11, the fp16
unit roundoff (4 u A).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import compare, oracle_decode, oracle_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


PREFILL = [
    (1, 2, 2, 128, 128, 64, False, None),
    (2, 4, 2, 300, 300, 128, True, None),
    (2, 4, 1, 200, 333, 128, True, (50, 333)),
    (2, 8, 2, 513, 513, 64, True, (200, 513)),
]


@pytest.mark.parametrize("case", PREFILL, ids=lambda c: "x".join(map(str, c[:6])) +
                         f"-c{int(c[6])}" + ("-pad" if c[7] else ""))
def test_prefill_f16(E, case):
    B, Hq, Hkv, T, S, D, causal, lens = case
    x = workloads.prefill_inputs(B, Hq, Hkv, T, S, D, "f16", seed=5, device="cuda", lens=lens)
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd(x["q"], x["k"], x["v"], causal=causal, key_lens=x["key_lens"],
                        scale=scale)
    torch.cuda.synchronize()
    assert o.dtype == torch.float16
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], causal, x["key_lens"], scale)
    compare(o, lse, ro, rl, torch.float16, f"f16 prefill {case}")
    assert E.attn_device_error(clear=True) == 0


def test_chunked_f16(E):
    B, Hq, Hkv, T, S_max, D = 2, 4, 2, 160, 700, 128
    g = torch.Generator(device="cuda").manual_seed(6)
    q = torch.randn(B, Hq, T, D, generator=g, device="cuda").half()
    kc = torch.randn(B, Hkv, S_max, D, generator=g, device="cuda").half()
    vc = torch.randn(B, Hkv, S_max, D, generator=g, device="cuda").half()
    qp = torch.tensor([300, 17], dtype=torch.int32, device="cuda")
    kl = torch.tensor([460, 100], dtype=torch.int32, device="cuda")
    for b in range(B):
        kc[b, :, int(kl[b]):] = float("nan")
        vc[b, :, int(kl[b]):] = float("nan")
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd_chunked(q, kc, vc, qp, kl, scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle_fwd(q, kc, vc, True, kl, scale, q_pos=qp)
    compare(o, lse, ro, rl, torch.float16, "f16 chunked")


@pytest.mark.parametrize("D,G", [(128, 4), (64, 1)])
def test_append_and_decode_f16(E, D, G):
    Hkv = 4
    d = workloads.decode_inputs(5, Hkv * G, Hkv, D, 100, 900, "f16", seed=7, device="cuda")
    E.kv_cache_append(d["kcache"], d["vcache"], d["k_new"], d["v_new"], d["cache_len"])
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_decode(d["q"], d["kcache"], d["vcache"], d["kv_len"], scale=scale)
    torch.cuda.synchronize()
    b_idx = torch.arange(5, device="cuda")
    assert torch.equal(d["kcache"][b_idx, :, d["cache_len"].long()], d["k_new"])
    assert torch.equal(d["vcache"][b_idx, :, d["cache_len"].long()], d["v_new"])
    ro, rl = oracle_decode(d["q"], d["kcache"], d["vcache"], d["kv_len"], scale)
    compare(o, lse, ro, rl, torch.float16, f"f16 decode D{D} G{G}")
    assert E.attn_device_error(clear=True) == 0


@pytest.mark.parametrize("D", [64, 128])
def test_backward_f16(E, D):
    B, Hq, Hkv, T, S = 2, 4, 2, 300, 300
    g = torch.Generator(device="cuda").manual_seed(8)
    q, k, v, do = (torch.randn(B, h, n, D, generator=g, device="cuda").half()
                   for h, n in ((Hq, T), (Hkv, S), (Hkv, S), (Hq, T)))
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd(q, k, v, causal=True, scale=scale)
    dq, dk, dv = E.attn_bwd(q, k, v, o, do, lse, causal=True, scale=scale)
    torch.cuda.synchronize()
    arrs = [t.cpu().numpy() for t in (q, k, v, do)]
    rq, rk, rv, _, _ = oracle.attn_bwd_np(*arrs, causal=True, scale=scale)
    mags = oracle.attn_bwd_magnitudes_np(*arrs, causal=True, scale=scale)
    u = 2.0 ** -11
    for name, got, ref, mag in (("dq", dq, rq, mags[0]), ("dk", dk, rk, mags[1]),
                                ("dv", dv, rv, mags[2])):
        gg = got.double().cpu().numpy()
        assert np.isfinite(gg).all()
        err = np.abs(gg - ref)
        assert (err <= 4 * u * mag).all(), f"{name}: beyond 4u A by {(err - 4 * u * mag).max():.3g}"
        assert np.linalg.norm(gg - ref) / np.linalg.norm(ref) <= 1e-2 / 4
    assert E.attn_device_error(clear=True) == 0
