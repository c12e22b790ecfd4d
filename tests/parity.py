"""Helpers for the GPU-vs-oracle parity tests.

Tolerances (float64 oracle as reference, same input values on both sides):
  float32 path: O max abs <= 2e-5, LSE max abs <= 1e-4
  bf16 path:    O max abs <= 1.5e-2 and mean abs <= 2e-3, LSE max abs <= 2e-3
  fp16 path:    the bf16 bounds x 1/4 (the unit-roundoff ratio 2^-11 / 2^-8
                is 1/8; a factor 2 of it is left for fp32 accumulation and
                ex2.approx)
Rows with no visible key (padded rows included) must be exactly O = 0 and
LSE = -inf on the GPU; they are excluded from the tolerance statistics.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import to_numpy_exact

TOL = {
    torch.float32: {"max": 2e-5, "mean": 2e-5, "lse": 1e-4},
    torch.bfloat16: {"max": 1.5e-2, "mean": 2e-3, "lse": 2e-3},
    # fp16 keeps 11 significant bits against bf16's 8: the errors come from
    # rounding P and O, whose unit roundoffs are in the ratio 2^-11 / 2^-8 =
    # 1/8; the bf16 bounds are scaled by 1/4, which leaves a factor 2 for the
    # fp32 accumulation and ex2.approx.
    torch.float16: {"max": 3.75e-3, "mean": 5e-4, "lse": 5e-4},
}


def oracle_fwd(q, k, v, causal, key_lens, scale, rows=None, q_pos=None):
    qn, bf = to_numpy_exact(q)
    kn, _ = to_numpy_exact(k)
    vn, _ = to_numpy_exact(v)
    kl = None if key_lens is None else key_lens.cpu().numpy()
    qp = None if q_pos is None else q_pos.cpu().numpy()
    return oracle.attn_fwd(qn, kn, vn, causal=causal, key_lens=kl, scale=scale,
                           bf16=bf, rows=rows, q_pos=qp)


def oracle_decode(q, kc, vc, kv_lens, scale):
    qn, bf = to_numpy_exact(q)
    kn, _ = to_numpy_exact(kc)
    vn, _ = to_numpy_exact(vc)
    return oracle.attn_decode(qn, kn, vn, kv_lens.cpu().numpy(), scale=scale, bf16=bf)


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bfloat16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.ldexp(1.0, np.floor(np.log2(ax)).astype(np.int64) - 8)


def compare(o_gpu: torch.Tensor, lse_gpu, o_ref: np.ndarray, lse_ref: np.ndarray,
            dtype, what="", out_rounding=False):
    """Element-by-element comparison; returns the error statistics.

    ``out_rounding`` widens the per-element max bound by half a bf16 ulp of
    the exact value: only for stress cases whose outputs exceed magnitude 2,
    where storing O in bf16 alone can cost up to 1.56e-2.
    """
    tol = TOL[dtype]
    og = o_gpu.detach().double().cpu().numpy().reshape(o_ref.shape)
    empty = ~np.isfinite(lse_ref)
    # Rows with no visible key: exact zeros (and -inf LSE) required.
    assert np.all(og[empty] == 0.0), f"{what}: rows without visible keys must be exactly 0"
    good = ~empty
    assert np.isfinite(og).all(), f"{what}: non-finite outputs"
    err = np.abs(og[good] - o_ref[good]) if good.any() else np.zeros(1)
    stats = {"max": float(err.max()), "mean": float(err.mean()), "rows": int(good.sum()),
             "empty_rows": int(empty.sum())}
    if out_rounding and good.any():
        excess = err - bf16_half_ulp(o_ref[good])
        assert excess.max() <= tol["max"], \
            f"{what}: max abs err beyond output rounding {excess.max():.3g} > {tol['max']}"
    else:
        assert stats["max"] <= tol["max"], f"{what}: max abs err {stats['max']:.3g} > {tol['max']}"
    assert stats["mean"] <= tol["mean"], f"{what}: mean abs err {stats['mean']:.3g} > {tol['mean']}"
    if lse_gpu is not None:
        lg = lse_gpu.detach().double().cpu().numpy().reshape(lse_ref.shape)
        assert np.all(lg[empty] == -np.inf), f"{what}: LSE of empty rows must be -inf"
        if good.any():
            le = np.abs(lg[good] - lse_ref[good])
            stats["lse_max"] = float(le.max())
            assert stats["lse_max"] <= tol["lse"], \
                f"{what}: LSE max abs err {stats['lse_max']:.3g} > {tol['lse']}"
    return stats


def sample_rows(B, Hq, T, S, lens, per_head, seed, q_off=None):
    """Flat row ids (b*Hq + h)*T + i to compare one by one: the first and
    last rows of each head, the rows around the first two tile boundaries,
    the rows at and after each sequence's valid length, and `per_head`
    seeded random rows per head."""
    rng = np.random.default_rng(seed)
    rows = []
    off = S - T if q_off is None else q_off
    for b in range(B):
        L = S if lens is None else int(lens[b])
        for h in range(Hq):
            base = (b * Hq + h) * T
            pick = {0, 1, 127, 128, 255, 256, T - 2, T - 1, max(L - off - 1, 0),
                    min(max(L - off, 0), T - 1)}
            pick |= set(rng.integers(0, T, size=per_head).tolist())
            rows.extend(base + i for i in sorted(pick) if 0 <= i < T)
    return np.array(rows, dtype=np.int64)


def gather_rows(o: torch.Tensor, lse: torch.Tensor, rows: np.ndarray, D: int):
    """The GPU outputs of the given flat rows: (o [n, D], lse [n])."""
    idx = torch.from_numpy(rows).to(o.device)
    return o.reshape(-1, D).index_select(0, idx), lse.reshape(-1).index_select(0, idx)


def assert_padded_rows_zero(o: torch.Tensor, lse: torch.Tensor, lens, S: int):
    """Every padded query row (position >= L_b, bottom-right alignment) is
    exactly 0 with LSE = -inf, and every other row has a finite LSE."""
    B, Hq, T, _ = o.shape
    for b in range(B):
        L = int(lens[b])
        first_pad = max(0, min(T, L - (S - T)))
        assert torch.all(o[b, :, first_pad:] == 0), f"padded rows of sequence {b} not zero"
        assert torch.all(torch.isneginf(lse[b, :, first_pad:]))
        assert torch.all(torch.isfinite(lse[b, :, :first_pad]))
