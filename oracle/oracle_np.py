"""NumPy float64 twin of the C oracle, and the tiled online-softmax recurrence.

TEST INFRASTRUCTURE ONLY: imported by tests, the smoke check and the
benchmark's CPU baseline, never by the product path.

``attn_fwd_np`` / ``attn_decode_np`` compute the same plain definition as
``attn_oracle.c`` but are written independently (vectorised NumPy, boolean
masks instead of per-key branches), so that the two can be compared.

``attn_tiled_online_np`` is the method itself, stated in float64: keys are
processed in tiles while a running row maximum ``m`` and denominator ``l`` are
kept, and earlier partial sums are rescaled by ``exp(m_old - m_new)`` whenever
the maximum grows ("Implementing attention from scratch", Core ideas, Stable
softmax; "Self-Attention: Implementation, Complexity, and Efficient
Variants", Task 2 and Hint 1; "FlashAttention", section 9.4.1 and Figure
9.8).  The NumPy build guide's Step 5 normalises each key tile on its own and
adds the tiles together, which does not give softmax; the recurrence here is
the reading its own Architecture Overview ("running max and sum of
exponentials") and the other pages support.  It is used only to check
"tiled == full", never as the oracle.
"""
from __future__ import annotations

import numpy as np

_NEG_INF = -np.inf


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of raw bfloat16 bit patterns (uint16) to float64."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def e4m3_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of FP8 E4M3 bit patterns (uint8) to float64.

    The format of the FP8 inputs that "Self-Attention: Implementation,
    Complexity, and Efficient Variants" (FlashAttention-3: FP8 support)
    refers to, as published in "FP8 Formats for Deep Learning" (Micikevicius
    et al., 2022) and the OCP 8-bit floating point specification: one sign
    bit, four exponent bits with bias 7, three mantissa bits; exponent field 0
    holds the subnormals m/8 * 2^-6; there are no infinities and S.1111.111 is
    NaN, so the largest finite magnitude is 1.75 * 2^8 = 448.
    """
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 0x7).astype(np.float64)
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    val = np.where((e == 0xF) & ((b & 0x7) == 0x7), np.nan, val)
    return sign * val


def attn_fwd_fp8_np(q8, k8, v8, q_descale=1.0, k_descale=1.0, v_descale=1.0, causal=False,
                    key_lens=None, scale=None):
    """Attention on FP8 E4M3 inputs: the plain definition of attn_fwd_np
    applied to the dequantised inputs q = q8 * q_descale, k = k8 * k_descale,
    v = v8 * v_descale (per-tensor scales, the FlashAttention-3 convention),
    in float64.  Returns (o, lse)."""
    q = e4m3_bits_to_f64(q8) * q_descale
    k = e4m3_bits_to_f64(k8) * k_descale
    v = e4m3_bits_to_f64(v8) * v_descale
    return attn_fwd_np(q, k, v, causal=causal, key_lens=key_lens, scale=scale)


def _as_f64(x: np.ndarray, bf16: bool) -> np.ndarray:
    if bf16:
        return bf16_bits_to_f64(np.asarray(x, dtype=np.uint16))
    return np.asarray(x, dtype=np.float64)


def visibility(T: int, S: int, L: int, causal: bool,
               q0: int | None = None) -> tuple[np.ndarray, np.ndarray]:
    """(row_valid [T], visible [T,S]) for one sequence.

    Query row i sits at key position q0 + i, where q0 = S - T by default
    (bottom-right alignment) or the cache length before the chunk (chunked
    prefill against a cache).  It is a padded row when that position is
    >= L.  Key j is visible to row i when j < L and, for causal attention,
    j <= q0 + i.
    """
    if q0 is None:
        q0 = S - T
    pos = np.arange(T)[:, None] + q0
    j = np.arange(S)[None, :]
    vis = j < L
    if causal:
        vis = vis & (j <= pos)
    row_valid = (np.arange(T) + q0) < L
    vis = vis & row_valid[:, None]
    return row_valid, vis


def attn_fwd_np(q, k, v, causal=False, key_lens=None, scale=None, bf16=False,
                q_pos=None):
    """Full-softmax attention in float64.  q [B,Hq,T,D], k/v [B,Hkv,S,D].

    ``q_pos`` ([B], optional) puts query row i of sequence b at key position
    q_pos[b] + i (chunked prefill); default S - T.  Returns (o [B,Hq,T,D],
    lse [B,Hq,T]); rows with no visible key (padded rows included) are O = 0,
    LSE = -inf.
    """
    q, k, v = (_as_f64(x, bf16) for x in (q, k, v))
    B, Hq, T, D = q.shape
    _, Hkv, S, _ = k.shape
    assert Hq % Hkv == 0
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    G = Hq // Hkv
    o = np.zeros((B, Hq, T, D))
    lse = np.full((B, Hq, T), _NEG_INF)
    for b in range(B):
        L = S if key_lens is None else int(key_lens[b])
        _, vis = visibility(T, S, L, causal, None if q_pos is None else int(q_pos[b]))
        # Masked-out scores are never formed: a key row outside the visible
        # set may hold anything (even NaN) without touching the result.
        has = vis.any(axis=1)
        for h in range(Hq):
            g = h // G
            with np.errstate(invalid="ignore"):
                s = (q[b, h] @ np.where(vis.any(axis=0)[:, None], k[b, g], 0.0).T) * scale
            s = np.where(vis, s, _NEG_INF)
            m = np.where(has, s.max(axis=1), 0.0)
            e = np.where(vis, np.exp(s - m[:, None]), 0.0)
            z = e.sum(axis=1)
            zs = np.where(has, z, 1.0)
            o[b, h] = (e / zs[:, None]) @ np.where(vis.any(axis=0)[:, None], v[b, g], 0.0)
            lse[b, h] = np.where(has, m + np.log(zs), _NEG_INF)
    return o, lse


def attn_decode_np(q, kcache, vcache, kv_lens, scale=None, bf16=False):
    """One query per (b, h) against the first kv_lens[b] cache rows.

    q [B,Hq,D], caches [B,Hkv,S_max,D].  Returns (o [B,Hq,D], lse [B,Hq]).
    """
    q4 = np.asarray(q)[:, :, None, :]
    q4 = _as_f64(q4, bf16)
    kc, vc = _as_f64(kcache, bf16), _as_f64(vcache, bf16)
    B, Hq, _, D = q4.shape
    o = np.zeros((B, Hq, D))
    lse = np.full((B, Hq), _NEG_INF)
    for b in range(B):
        L = int(kv_lens[b])
        if L <= 0:
            continue
        # The single query sits at position L-1 and sees keys 0..L-1.
        ob, lb = attn_fwd_np(q4[b:b + 1], kc[b:b + 1, :, :L], vc[b:b + 1, :, :L],
                             causal=True, key_lens=None, scale=scale)
        o[b] = ob[0, :, 0]
        lse[b] = lb[0, :, 0]
    return o, lse


def attn_tiled_online_np(q, k, v, causal=False, key_lens=None, scale=None,
                         tile_q=64, tile_k=64, bf16=False):
    """The tiled method with an online softmax, in float64.

    For every query tile, keys are visited tile by tile.  Per row it keeps the
    running maximum m, the running denominator l and the unnormalised output
    acc.  With the scores s of a new key tile:

        m_new = max(m, rowmax(s))
        acc   = acc * exp(m - m_new) + exp(s - m_new) @ V_tile
        l     = l   * exp(m - m_new) + rowsum(exp(s - m_new))

    and at the end O = acc / l, LSE = m + ln l.
    """
    q, k, v = (_as_f64(x, bf16) for x in (q, k, v))
    B, Hq, T, D = q.shape
    _, Hkv, S, _ = k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    G = Hq // Hkv
    o = np.zeros((B, Hq, T, D))
    lse = np.full((B, Hq, T), _NEG_INF)
    for b in range(B):
        L = S if key_lens is None else int(key_lens[b])
        _, vis = visibility(T, S, L, causal)
        for h in range(Hq):
            g = h // G
            for q0 in range(0, T, tile_q):
                q1 = min(q0 + tile_q, T)
                n = q1 - q0
                m = np.full(n, _NEG_INF)
                l = np.zeros(n)
                acc = np.zeros((n, D))
                for k0 in range(0, S, tile_k):
                    k1 = min(k0 + tile_k, S)
                    s = (q[b, h, q0:q1] @ k[b, g, k0:k1].T) * scale
                    tv = vis[q0:q1, k0:k1]
                    s = np.where(tv, s, _NEG_INF)
                    m_new = np.maximum(m, s.max(axis=1))
                    # Rows that have seen no visible key yet keep a zero
                    # reference so that exp() of -inf - -inf never appears.
                    ref = np.where(np.isfinite(m_new), m_new, 0.0)
                    alpha = np.where(np.isfinite(m), np.exp(m - ref), 0.0)
                    p = np.where(tv, np.exp(s - ref[:, None]), 0.0)
                    acc = acc * alpha[:, None] + p @ v[b, g, k0:k1]
                    l = l * alpha + p.sum(axis=1)
                    m = m_new
                has = l > 0
                ls = np.where(has, l, 1.0)
                o[b, h, q0:q1] = np.where(has[:, None], acc / ls[:, None], 0.0)
                lse[b, h, q0:q1] = np.where(has, m + np.log(ls), _NEG_INF)
    return o, lse


def attn_bwd_np(q, k, v, do, causal=False, key_lens=None, scale=None, bf16=False,
                q_pos=None):
    """Gradients of attention in float64: (dq, dk, dv), plus (o, lse).

    The chain rule through the softmax, written out step by step for each
    (b, h) with g = h / (Hq / Hkv).  Sources: "Hands-on build guide:
    FlashAttention-style tiled attention kernel in pure NumPy", Roadmap
    (gradient through attention: dL/dQ, dL/dK, dL/dV by the chain rule);
    "Self-Attention: Implementation, Complexity, and Efficient Variants",
    FlashAttention follow-up (the backward pass recomputes the attention
    matrix on chip instead of storing it); "Implementing attention from
    scratch", Testing against a reference (gradient comparisons against a
    float64 reference).  This function is that reference:

        S  = scale * Q K^T            (visible entries only)
        P  = softmax_rows(S)          (0 on hidden keys; rows with no
                                       visible key are all 0)
        O  = P V
        dV = P^T dO                   (summed over the Hq/Hkv heads of g)
        dP = dO V^T
        Δ  = rowsum(dO * O)           (= rowsum(P * dP))
        dS = P * (dP - Δ)
        dQ = scale * dS K
        dK = scale * dS^T Q           (summed over the heads of g)

    q, do [B,Hq,T,D]; k, v [B,Hkv,S,D]; masks and q_pos as in attn_fwd_np.
    """
    q, k, v, do = (_as_f64(x, bf16) for x in (q, k, v, do))
    B, Hq, T, D = q.shape
    _, Hkv, S, _ = k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    G = Hq // Hkv
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    o = np.zeros_like(q)
    lse = np.full((B, Hq, T), _NEG_INF)
    for b in range(B):
        L = S if key_lens is None else int(key_lens[b])
        _, vis = visibility(T, S, L, causal, None if q_pos is None else int(q_pos[b]))
        has = vis.any(axis=1)
        keys = vis.any(axis=0)
        for h in range(Hq):
            g = h // G
            kg = np.where(keys[:, None], k[b, g], 0.0)
            vg = np.where(keys[:, None], v[b, g], 0.0)
            s = np.where(vis, (q[b, h] @ kg.T) * scale, _NEG_INF)
            m = np.where(has, s.max(axis=1), 0.0)
            e = np.where(vis, np.exp(s - m[:, None]), 0.0)
            z = np.where(has, e.sum(axis=1), 1.0)
            p = e / z[:, None]
            o[b, h] = p @ vg
            lse[b, h] = np.where(has, m + np.log(z), _NEG_INF)
            dv[b, g] += p.T @ do[b, h]
            dp = do[b, h] @ vg.T
            delta = (do[b, h] * o[b, h]).sum(axis=1)
            ds = p * (dp - delta[:, None])
            dq[b, h] = scale * (ds @ kg)
            dk[b, g] += scale * (ds.T @ q[b, h])
    return dq, dk, dv, o, lse


def attn_bwd_magnitudes_np(q, k, v, do, causal=False, key_lens=None, scale=None, bf16=False,
                           q_pos=None):
    """Per-element magnitudes that bound the rounding error of a bf16
    evaluation of the backward (test infrastructure for tolerances).

    With u the unit roundoff of one rounding (2^-8 for bf16: half the spacing
    2^-7 of bf16 numbers on [1, 2); 2^-11 for fp16), a kernel that rounds P
    and dS to bf16
    before the products, forms delta from the bf16-rounded O and rounds
    each result once has, to first order, an error of at most u times:

        A_dq = scale * (|dS| |K| + (P |K|) * rowsum(|dO * O|)) + |dQ|
        A_dk = scale * (|dS|^T |Q| + P^T (|Q| * rowsum(|dO * O|))) + |dK|
        A_dv = P^T |dO| + |dV|

    (the first terms: rounding of dS; the second: the error of delta,
    rowsum(dO * O) with O rounded; the last: rounding of the result).
    Returns (A_dq, A_dk, A_dv) in the shapes of dq, dk, dv.
    """
    q, k, v, do = (_as_f64(x, bf16) for x in (q, k, v, do))
    B, Hq, T, D = q.shape
    _, Hkv, S, _ = k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    G = Hq // Hkv
    aq = np.zeros_like(q)
    ak = np.zeros_like(k)
    av = np.zeros_like(v)
    dq, dk, dv, o, _ = attn_bwd_np(q, k, v, do, causal=causal, key_lens=key_lens, scale=scale,
                                   q_pos=q_pos)
    for b in range(B):
        L = S if key_lens is None else int(key_lens[b])
        _, vis = visibility(T, S, L, causal, None if q_pos is None else int(q_pos[b]))
        has = vis.any(axis=1)
        keys = vis.any(axis=0)
        for h in range(Hq):
            g = h // G
            kg = np.where(keys[:, None], k[b, g], 0.0)
            vg = np.where(keys[:, None], v[b, g], 0.0)
            s = np.where(vis, (q[b, h] @ kg.T) * scale, _NEG_INF)
            m = np.where(has, s.max(axis=1), 0.0)
            e = np.where(vis, np.exp(s - m[:, None]), 0.0)
            p = e / np.where(has, e.sum(axis=1), 1.0)[:, None]
            dp = do[b, h] @ vg.T
            delta = (do[b, h] * o[b, h]).sum(axis=1)
            ads = np.abs(p * (dp - delta[:, None]))
            rdo = np.abs(do[b, h] * o[b, h]).sum(axis=1)          # rowsum |dO * O|
            aq[b, h] = scale * (ads @ np.abs(kg) + (p @ np.abs(kg)) * rdo[:, None])
            ak[b, g] += scale * (ads.T @ np.abs(q[b, h]) + p.T @ (np.abs(q[b, h]) * rdo[:, None]))
            av[b, g] += p.T @ np.abs(do[b, h])
    return aq + np.abs(dq), ak + np.abs(dk), av + np.abs(dv)


def attn_fwd_kv_shard_np(q, k, v, q_pos, key_lens, k_off, causal=True, scale=None, bf16=False):
    """Attention of the queries over one shard of the keys, in float64.

    "Building a causal self-attention block from scratch in PyTorch",
    Extending It: distributed attention shards Q/K/V across devices and
    recombines the results.  k, v [B,Hkv,S,D] hold the keys at global
    positions k_off .. k_off + S - 1 of each sequence.  In global positions:
    query row i of sequence b sits at q_pos[b] + i; key x is visible to it
    iff x < key_lens[b] and (not causal, or x <= q_pos[b] + i); the row is
    a padded row iff q_pos[b] + i >= key_lens[b].  The result is the
    softmax over the visible keys of this shard only, with its LSE: (o
    [B,Hq,T,D], lse [B,Hq,T]); rows that see no key of the shard (padded
    rows included) are O = 0, LSE = -inf.
    """
    q, k, v = (_as_f64(x, bf16) for x in (q, k, v))
    B, Hq, T, D = q.shape
    _, Hkv, S, _ = k.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    G = Hq // Hkv
    o = np.zeros((B, Hq, T, D))
    lse = np.full((B, Hq, T), _NEG_INF)
    x = k_off + np.arange(S)                       # global key positions
    for b in range(B):
        L = int(key_lens[b])
        pos = int(q_pos[b]) + np.arange(T)         # global query positions
        vis = (x[None, :] < L) & (pos[:, None] < L)
        if causal:
            vis &= x[None, :] <= pos[:, None]
        for h in range(Hq):
            g = h // G
            for i in range(T):
                j = np.nonzero(vis[i])[0]
                if j.size == 0:
                    continue
                s = scale * (k[b, g, j] @ q[b, h, i])
                m = s.max()
                e = np.exp(s - m)
                o[b, h, i] = (e / e.sum()) @ v[b, g, j]
                lse[b, h, i] = m + np.log(e.sum())
    return o, lse


def lse_merge_np(o_parts, lse_parts):
    """Attention over the union of disjoint key sets from the partials over
    each set, in float64: with Z_n = exp(LSE_n) the sum of exponentials of
    part n and O_n its normalised output, the whole row has
    Z = sum_n Z_n and O = sum_n Z_n O_n / Z ("Implementing attention from
    scratch", Core ideas, Stable softmax: the same rescaling the online
    softmax applies).  Computed against the largest LSE_n of the row; a row
    with no finite LSE_n is O = 0, LSE = -inf.  o_parts [N,...,D],
    lse_parts [N,...] -> (o [...,D], lse [...])."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    finite = np.isfinite(lse_parts)
    m = np.where(finite, lse_parts, _NEG_INF).max(axis=0)
    has = np.isfinite(m)
    ref = np.where(has, m, 0.0)
    w = np.where(finite, np.exp(np.where(finite, lse_parts, 0.0) - ref[None]), 0.0)
    z = w.sum(axis=0)
    zs = np.where(has, z, 1.0)
    o = np.where(has[..., None], (w[..., None] * np.nan_to_num(o_parts)).sum(axis=0)
                 / zs[..., None], 0.0)
    lse = np.where(has, ref + np.log(zs), _NEG_INF)
    return o, lse
