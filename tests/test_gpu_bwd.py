"""GPU parity of the attention backward (attn_bwd) with the float64 oracle.

The forward's O and LSE come from the GPU (as in training); the oracle
recomputes everything in float64 from the same bf16 inputs.

Tolerance (derived, not fitted): bf16 keeps 8 significant bits, so one
rounding costs at most u = 2^-8 of the value (half the spacing 2^-7 of
bf16 numbers on [1, 2)).  The GPU rounds P and dS to
bf16 before the products (fp32 accumulation), forms delta = rowsum(dO * O)
from the forward's bf16-rounded O, and rounds each result once.  To first
order the error of every element is then at most u times a magnitude the
oracle computes in float64 (oracle.attn_bwd_magnitudes_np: the sums of
absolute terms that each rounding perturbs; the delta term matters where
dP - delta nearly cancels, as in the first rows of a causal mask).  The
tests require

    elementwise |g - g_ref| <= 2 u A        (2: fp32 accumulation, ex2.approx,
                                             second-order terms, and the forward's
                                             O carrying more than one rounding)
    normwise    ||g - g_ref|| / ||g_ref||  <= 1e-2

Rows that see no key must have dQ exactly 0; keys no row sees, dK = dV = 0.
Cases cover ragged tiles, GQA, T < S and T > S, key padding (padded K/V rows
hold NaN), non-causal, chunked query positions, D in {64, 128}.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from workloads import to_numpy_exact

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


def check_grad(g_gpu, g_ref, mag, name):
    g = g_gpu.detach().double().cpu().numpy()
    assert np.isfinite(g).all(), f"{name}: non-finite values"
    err = np.abs(g - g_ref)
    nref = np.linalg.norm(g_ref)
    if nref > 0:
        rel = np.linalg.norm(g - g_ref) / nref
        assert rel <= 1e-2, f"{name}: normwise relative error {rel:.3g}"
    bound = 2.0 * 2.0 ** -8 * mag    # 2 u A, u = 2^-8 the bf16 unit roundoff
    worst = float((err - bound).max())
    assert worst <= 0, f"{name}: elementwise error beyond bound by {worst:.3g} (max err {err.max():.3g})"
    return float(err.max())


CASES = [
    # (B, Hq, Hkv, T, S, D, causal, key_lens, q_pos)
    (1, 2, 2, 128, 128, 64, False, None, None),
    (2, 4, 2, 300, 300, 128, True, None, None),
    (2, 2, 2, 200, 333, 64, True, [150, 333], None),
    (1, 2, 1, 333, 200, 128, True, None, None),
    (2, 4, 4, 257, 513, 128, False, [513, 100], None),
    (2, 4, 2, 100, 400, 64, True, [300, 150], [200, 50]),
    (1, 8, 2, 640, 640, 128, True, [640], None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + f"-c{int(c[6])}"
                         + ("-pad" if c[7] else "") + ("-qpos" if c[8] else ""))
def test_backward(E, case):
    B, Hq, Hkv, T, S, D, causal, lens, qpos = case
    g = torch.Generator(device="cuda").manual_seed(41)
    q = torch.randn(B, Hq, T, D, generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, Hkv, S, D, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(B, Hkv, S, D, generator=g, device="cuda").to(torch.bfloat16)
    dout = torch.randn(B, Hq, T, D, generator=g, device="cuda").to(torch.bfloat16)
    kl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    qp = None if qpos is None else torch.tensor(qpos, dtype=torch.int32, device="cuda")
    if kl is not None:
        for b in range(B):   # rows past the valid length may hold anything
            k[b, :, int(kl[b]):] = float("nan")
            v[b, :, int(kl[b]):] = float("nan")
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
    rq, rk, rv, _, rl = oracle.attn_bwd_np(
        *bits, causal=causal, key_lens=None if kl is None else kl.cpu().numpy(), scale=scale,
        bf16=True, q_pos=None if qp is None else qp.cpu().numpy())
    aq, ak, av = oracle.attn_bwd_magnitudes_np(
        *bits, causal=causal, key_lens=None if kl is None else kl.cpu().numpy(), scale=scale,
        bf16=True, q_pos=None if qp is None else qp.cpu().numpy())
    check_grad(dq, rq, aq, "dq")
    check_grad(dk, rk, ak, "dk")
    check_grad(dv, rv, av, "dv")
    # structure: rows that see nothing have dQ = 0; unseen keys have dK = dV = 0
    empty = ~np.isfinite(rl)
    assert np.all(dq.double().cpu().numpy()[empty] == 0)
    unseen = np.all(rk == 0, axis=-1) & np.all(rv == 0, axis=-1)
    assert np.all(dk.double().cpu().numpy()[unseen] == 0)
    assert np.all(dv.double().cpu().numpy()[unseen] == 0)


def test_backward_rejects_bad_arguments(E):
    x = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(1, 1, 128, device="cuda")
    with pytest.raises(E.AttnError):   # fp32 takes D <= 256
        xf = torch.zeros(1, 1, 128, 260, device="cuda")
        E.attn_bwd(xf, xf, xf, xf, xf, lse)
    with pytest.raises(E.AttnError):   # D must be 64 or 128
        y = torch.zeros(1, 1, 128, 32, dtype=torch.bfloat16, device="cuda")
        E.attn_bwd(y, y, y, y, y, lse)
    with pytest.raises(E.AttnError):   # workspace too small
        E.attn_bwd(x, x, x, x, x, lse, workspace=torch.empty(16, dtype=torch.uint8, device="cuda"))


F32_CASES = [
    # (B, Hq, Hkv, T, S, D, causal, key_lens, q_pos)
    (2, 4, 2, 130, 200, 64, True, [200, 77], None),
    (1, 2, 1, 100, 300, 37, False, [250], None),
    (2, 2, 2, 150, 150, 128, True, None, [10, -20]),
    (1, 8, 2, 90, 90, 256, True, None, None),
    (2, 3, 3, 33, 65, 1, True, [65, 0], None),
]


@pytest.mark.parametrize("case", F32_CASES, ids=lambda c: "x".join(map(str, c[:6])))
def test_backward_fp32(E, case):
    """The exact fp32 backward (CUDA cores).  Bound, derived: with fp32's unit
    roundoff u = 2^-24, dot products of D terms and sums over at most n rows
    or keys with fused multiply-adds, the forward's fp32 O and LSE, and
    accurate expf (a few ulp), every element is within 4 (D + n) u A of the
    float64 result, A the sum of absolute terms (oracle.attn_bwd_magnitudes_np);
    normwise 1e-5."""
    B, Hq, Hkv, T, S, D, causal, lens, qpos = case
    g = torch.Generator(device="cuda").manual_seed(43)
    q = torch.randn(B, Hq, T, D, generator=g, device="cuda")
    k = torch.randn(B, Hkv, S, D, generator=g, device="cuda")
    v = torch.randn(B, Hkv, S, D, generator=g, device="cuda")
    dout = torch.randn(B, Hq, T, D, generator=g, device="cuda")
    kl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    qp = None if qpos is None else torch.tensor(qpos, dtype=torch.int32, device="cuda")
    if kl is not None:
        for b in range(B):   # rows past the valid length may hold anything
            k[b, :, int(kl[b]):] = float("nan")
            v[b, :, int(kl[b]):] = float("nan")
    scale = 1.0 / math.sqrt(D)
    if qp is None:
        o, lse = E.attn_fwd(q, k, v, causal=causal, key_lens=kl, scale=scale)
    else:
        klc = kl if kl is not None else torch.full((B,), S, dtype=torch.int32, device="cuda")
        o, lse = E.attn_fwd_chunked(q, k, v, qp, klc, causal=causal, scale=scale)
    dq, dk, dv = E.attn_bwd(q, k, v, o, dout, lse, causal=causal, key_lens=kl, q_pos=qp,
                            scale=scale)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    arr = [t.cpu().numpy() for t in (q, k, v, dout)]
    kw = dict(causal=causal, key_lens=None if kl is None else kl.cpu().numpy(), scale=scale,
              bf16=False, q_pos=None if qp is None else qp.cpu().numpy())
    rq, rk, rv, _, rl = oracle.attn_bwd_np(*arr, **kw)
    aq, ak, av = oracle.attn_bwd_magnitudes_np(*arr, **kw)
    n = max(S, T * (Hq // Hkv))
    for gg, ref, mag, name in ((dq, rq, aq, "dq"), (dk, rk, ak, "dk"), (dv, rv, av, "dv")):
        x = gg.double().cpu().numpy()
        assert np.isfinite(x).all(), name
        err = np.abs(x - ref)
        assert (err <= 4 * (D + n) * 2.0 ** -24 * mag + 1e-30).all(), \
            f"{name}: max err {err.max():.3g}"
        nref = np.linalg.norm(ref)
        if nref > 0:
            assert np.linalg.norm(x - ref) / nref <= 1e-5, name
    empty = ~np.isfinite(rl)
    assert np.all(dq.double().cpu().numpy()[empty] == 0)
