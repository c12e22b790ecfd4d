"""Seeded synthetic inputs shared by the tests, the smoke check and bench.py.

This module only draws random numbers and lays them out; it holds none of
the attention arithmetic.  Both the CUDA path and the oracle are fed from it.

Workloads (sizes follow the pages' examples and the benchmark shapes):

1. single-head non-causal fp32: Q n=256 x d=64, K/V m=512 x d=64, drawn with
   ``np.random.seed(0)`` then ``randn`` for Q, K, V in that order, exactly as
   in "Hands-on build guide: FlashAttention-style tiled attention kernel in
   pure NumPy", Step 1; scale 1/sqrt(64).
2. causal self-attention prefill: B=4, H=8, T=S=1024, D=64, bf16.
3. long-context causal prefill: B=1, H=16, T=S=32768, D=128, bf16, Q = 2 x.
4. GQA KV-cache decode: B=64, Hq=32, Hkv=8, D=128, bf16, cache length per
   sequence uniform in [1024, 8192]; the new token is appended at offset
   cache_len and attends over cache_len + 1 keys.
5. padded batch prefill: B=8, H=16, T=S=4096, D=128, bf16, causal, valid
   length per sequence uniform in [2048, 4096].

Recipe for workloads 2-5 and for every other seeded case: a
``torch.Generator`` on the target device seeded with the workload id (or the
given seed) draws N(0, 1) float32 values in the order q, k, v (decode: q,
kcache, vcache, k_new, v_new); bf16 tensors are the round-to-nearest-even
casts of those values; "Q scaled by 2" multiplies the bf16 values by 2, which
is exact.  Lengths come from ``numpy.random.default_rng(seed).integers(lo,
hi + 1, size=B)`` (inclusive uniform).  The same seed gives different values
on the CPU and CUDA generators, so a test draws on one device and copies.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    wid: int
    name: str
    kind: str                  # "prefill" or "decode"
    dtype: str                 # "f32" or "bf16"
    B: int
    Hq: int
    Hkv: int
    D: int
    T: int = 0                 # prefill query length
    S: int = 0                 # prefill key length
    causal: bool = False
    lens: tuple | None = None  # (lo, hi) inclusive: key_lens / cache_len
    q_scale: float = 1.0
    extra: dict = field(default_factory=dict)


WORKLOADS = {
    1: Workload(1, "single-head non-causal attention fp32 n=256 m=512 d=64",
                "prefill", "f32", B=1, Hq=1, Hkv=1, D=64, T=256, S=512,
                causal=False),
    2: Workload(2, "causal self-attention prefill B=4 H=8 T=S=1024 D=64 bf16",
                "prefill", "bf16", B=4, Hq=8, Hkv=8, D=64, T=1024, S=1024,
                causal=True),
    3: Workload(3, "long-context causal prefill B=1 H=16 T=S=32768 D=128 bf16 Qx2",
                "prefill", "bf16", B=1, Hq=16, Hkv=16, D=128, T=32768,
                S=32768, causal=True, q_scale=2.0),
    4: Workload(4, "GQA KV-cache decode B=64 Hq=32 Hkv=8 D=128 bf16 cache_len U[1024,8192]",
                "decode", "bf16", B=64, Hq=32, Hkv=8, D=128,
                lens=(1024, 8192)),
    5: Workload(5, "padded batch causal prefill B=8 H=16 T=S=4096 D=128 bf16 key_len U[2048,4096]",
                "prefill", "bf16", B=8, Hq=16, Hkv=16, D=128, T=4096,
                S=4096, causal=True, lens=(2048, 4096)),
}

_DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def lengths(seed: int, lo: int, hi: int, B: int) -> np.ndarray:
    """Inclusive uniform integer lengths in [lo, hi], one per sequence."""
    return np.random.default_rng(seed).integers(lo, hi + 1, size=B).astype(np.int32)


def _randn(gen, shape, device, dtype, scale=1.0):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    x = x.to(_DT[dtype])
    if scale != 1.0:
        x = x * scale
    return x


def prefill_inputs(B, Hq, Hkv, T, S, D, dtype="bf16", seed=0, device="cpu",
                   q_scale=1.0, lens=None):
    """q [B,Hq,T,D], k/v [B,Hkv,S,D] and optional key_lens (int32 [B]).

    ``lens`` is None (every key valid) or an inclusive (lo, hi) range.
    """
    gen = torch.Generator(device=device).manual_seed(seed)
    q = _randn(gen, (B, Hq, T, D), device, dtype, q_scale)
    k = _randn(gen, (B, Hkv, S, D), device, dtype)
    v = _randn(gen, (B, Hkv, S, D), device, dtype)
    key_lens = None
    if lens is not None:
        key_lens = torch.from_numpy(lengths(seed, lens[0], lens[1], B)).to(device)
    return {"q": q, "k": k, "v": v, "key_lens": key_lens}


def decode_inputs(B, Hq, Hkv, D, lo, hi, dtype="bf16", seed=0, device="cpu",
                  s_max=None):
    """A KV cache with per-sequence lengths in [lo, hi] and one new token.

    Returns q [B,Hq,D], kcache/vcache [B,Hkv,S_max,D] (S_max = hi + 1 unless
    given), k_new/v_new [B,Hkv,D], cache_len (int32 [B], the append offset)
    and kv_len = cache_len + 1 (int32 [B]).
    """
    s_max = hi + 1 if s_max is None else s_max
    gen = torch.Generator(device=device).manual_seed(seed)
    q = _randn(gen, (B, Hq, D), device, dtype)
    kc = _randn(gen, (B, Hkv, s_max, D), device, dtype)
    vc = _randn(gen, (B, Hkv, s_max, D), device, dtype)
    kn = _randn(gen, (B, Hkv, D), device, dtype)
    vn = _randn(gen, (B, Hkv, D), device, dtype)
    cache_len = torch.from_numpy(lengths(seed, lo, hi, B)).to(device)
    return {"q": q, "kcache": kc, "vcache": vc, "k_new": kn, "v_new": vn,
            "cache_len": cache_len, "kv_len": cache_len + 1, "S_max": s_max}


def workload(wid: int, batch: int | None = None) -> Workload:
    """Workload `wid`, optionally with a smaller batch (a profiling case: the
    same shapes per sequence, fewer sequences)."""
    w = WORKLOADS[wid]
    if batch is None or batch == w.B:
        return w
    return replace(w, B=int(batch), name=f"{w.name} [profiling case: B={int(batch)}]")


def workload_inputs(wid: int, device="cpu", batch: int | None = None):
    """Inputs of one of the five named workloads, seeded with its id."""
    w = workload(wid, batch)
    if wid == 1:
        rs = np.random.RandomState(0)
        Q = rs.randn(w.T, w.D).astype(np.float32)
        K = rs.randn(w.S, w.D).astype(np.float32)
        V = rs.randn(w.S, w.D).astype(np.float32)
        t = lambda a: torch.from_numpy(a)[None, None].contiguous().to(device)
        return {"q": t(Q), "k": t(K), "v": t(V), "key_lens": None}
    if w.kind == "prefill":
        return prefill_inputs(w.B, w.Hq, w.Hkv, w.T, w.S, w.D, w.dtype,
                              seed=wid, device=device, q_scale=w.q_scale,
                              lens=w.lens)
    return decode_inputs(w.B, w.Hq, w.Hkv, w.D, w.lens[0], w.lens[1],
                         w.dtype, seed=wid, device=device)


def to_numpy_exact(t: torch.Tensor):
    """(array, is_bf16): float16/float32/float64 as is (NumPy widens them
    exactly), bf16 as raw uint16 bits."""
    t = t.detach().to("cpu").contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), True
    return t.numpy(), False
