"""GPU parity of the FP8 (E4M3) prefill (attn_fwd_fp8) with the float64 oracle.

The oracle (oracle.attn_fwd_fp8_np) is the plain definition on the
dequantised inputs.  Tolerance, derived from what the kernel rounds:

* scores: products of E4M3 values are exact in fp32 and accumulate in fp32
  (error ~2^-24 relative, negligible here);
* the softmax weights P' = 2^7 p (p relative to the running reference) are
  rounded to E4M3 for P V: relative error <= 2^-4 in the normal range, and
  at most 2^-10 absolute below it; the row sum l' >= 2^7 (the largest P' is
  at least 2^7), so a normalised weight w_j moves by at most
  2^-4 w_j + 2^-17;
* O is rounded once to bf16 (2^-9 relative).

Hence |o - o_ref| <= v_descale * sum_j (2^-4 w_j + 2^-17) |v8_j| + 2^-9 |o_ref|
per element; the test allows 1.25x that plus 1e-6 (ex2.approx, fp32
accumulation).  The LSE comes from unrounded fp32 weights: |dLSE| <= 2e-3.
Padded rows must be exactly O = 0, LSE = -inf.  Cases cover ragged tiles,
GQA, causal and not, key padding whose padded K/V bytes are NaN codes.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


def _fp8(x: torch.Tensor, descale: float) -> torch.Tensor:
    return (x / descale).to(torch.float8_e4m3fn)


CASES = [
    # (B, Hq, Hkv, T, S, causal, key_lens)
    (1, 1, 1, 128, 128, False, None),
    (1, 2, 2, 256, 256, True, None),
    (2, 4, 2, 300, 300, True, None),
    (2, 4, 1, 200, 333, True, (150, 333)),
    (1, 2, 2, 333, 200, False, None),
    (3, 4, 4, 640, 640, True, (0, 640, 257)),
    (1, 2, 1, 77, 1000, False, None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:5])) + f"-c{int(c[5])}"
                         + ("-pad" if c[6] else ""))
def test_fp8_prefill(E, case):
    B, Hq, Hkv, T, S, causal, lens = case
    D = 128
    qd, kd, vd = 0.25, 0.5, 0.125
    g = torch.Generator(device="cuda").manual_seed(81)
    q = _fp8(torch.randn(B, Hq, T, D, generator=g, device="cuda"), qd)
    k = _fp8(torch.randn(B, Hkv, S, D, generator=g, device="cuda"), kd)
    v = _fp8(torch.randn(B, Hkv, S, D, generator=g, device="cuda"), vd)
    kl = None
    if lens is not None:
        kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
        kb, vb = k.view(torch.uint8), v.view(torch.uint8)
        for b in range(B):  # padded rows may hold anything: E4M3 NaN codes here
            kb[b, :, lens[b]:] = 0x7F
            vb[b, :, lens[b]:] = 0x7F
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd_fp8(q, k, v, causal=causal, key_lens=kl, scale=scale,
                            q_descale=qd, k_descale=kd, v_descale=vd)
    torch.cuda.synchronize()
    assert E.attn_device_error(clear=True) == 0
    q8, k8, v8 = (t.view(torch.uint8).cpu().numpy() for t in (q, k, v))
    lens_np = None if kl is None else kl.cpu().numpy()
    ro, rl = oracle.attn_fwd_fp8_np(q8, k8, v8, qd, kd, vd, causal=causal, key_lens=lens_np,
                                    scale=scale)
    # bound terms from the same definition: weights applied to |v|, and sum of |v| seen
    vq = oracle.e4m3_bits_to_f64(q8) * qd
    vk = oracle.e4m3_bits_to_f64(k8) * kd
    av = np.abs(np.nan_to_num(oracle.e4m3_bits_to_f64(v8))) * vd
    wa, _ = oracle.attn_fwd_np(vq, vk, av, causal=causal, key_lens=lens_np, scale=scale)
    G = Hq // Hkv
    usum = np.zeros_like(ro)
    for b in range(B):
        L = S if lens_np is None else int(lens_np[b])
        _, vis = oracle.visibility(T, S, L, causal)
        for h in range(Hq):
            usum[b, h] = vis.astype(np.float64) @ av[b, h // G]
    bound = 1.25 * (2.0 ** -4 * wa + 2.0 ** -17 * usum + 2.0 ** -9 * np.abs(ro)) + 1e-6
    got = o.double().cpu().numpy()
    gl = lse.double().cpu().numpy()
    valid = np.isfinite(rl)
    assert np.isfinite(got).all()
    err = np.abs(got - ro)
    assert np.all(err[valid] <= bound[valid]), f"max excess {(err - bound)[valid].max():.3g}"
    assert np.all(got[~valid] == 0) and np.all(np.isneginf(gl[~valid]))
    assert np.abs(gl[valid] - rl[valid]).max() <= 2e-3
    # the bound is not vacuous: errors are a few percent of |v| at most
    assert err[valid].max() < 0.2 * np.abs(ro[valid]).max() + 0.05


def test_fp8_rejects_bad_arguments(E):
    q = torch.zeros(1, 1, 128, 64, dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(E.AttnError) as ex:
        E.attn_fwd_fp8(q, q, q)   # D = 64 is not supported
    assert ex.value.status == E.ATTN_ERR_UNSUPPORTED
    q = torch.zeros(1, 1, 128, 128, dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(E.AttnError) as ex:
        E.attn_fwd_fp8(q, q, q, v_descale=0.0)
    assert ex.value.status == E.ATTN_ERR_INVALID_ARG
