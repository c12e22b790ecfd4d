"""Pins for the float64 oracle (CPU only).

The oracle is the plain definition of attention ("Implementing attention
from scratch", Core ideas; "Building a causal self-attention block from
scratch in PyTorch", Steps 2-3).  Nothing here re-types that formula and
compares it with itself.  Instead every pin checks a fact that the pages or
mathematics fix independently:

* closed forms: Q = 0 makes every visible score equal, so O is the mean of
  the visible value rows and LSE = ln(#visible); two keys give a logistic
  weight; one key gives V[0];
* invariants: the weights are a convex combination (V = identity exposes
  them), identical value rows are reproduced, shifting every key by the same
  vector or permuting keys (non-causal) leaves O unchanged, GQA equals MHA
  with the KV heads repeated;
* the method: the tiled online-softmax recurrence equals the full softmax;
  incremental decoding equals the full causal forward at every step
  ("Implementing attention from scratch", Testing against a reference);
* a library special case: torch's float64 scaled_dot_product_attention with
  an explicit boolean mask ("Building a causal self-attention block",
  Running and Testing It).

``test_pins_catch_planted_mistakes`` plants plausible mistakes (a dropped
scale, a top-left causal mask, an off-by-one, the wrong softmax axis, the
wrong GQA mapping, ...) in a small CPU copy of the definition and checks that
each one fails at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ATOL = 1e-12


# --------------------------------------------------------------- adapters

def c_fwd(q, k, v, causal=False, key_lens=None, scale=None):
    return oracle.attn_fwd(q, k, v, causal=causal, key_lens=key_lens,
                           scale=scale, nthreads=2)


def np_fwd(q, k, v, causal=False, key_lens=None, scale=None):
    return oracle.attn_fwd_np(q, k, v, causal=causal, key_lens=key_lens,
                              scale=scale)


def c_dec(q, kc, vc, kv_lens, scale=None):
    return oracle.attn_decode(q, kc, vc, kv_lens, scale=scale, nthreads=2)


def np_dec(q, kc, vc, kv_lens, scale=None):
    return oracle.attn_decode_np(q, kc, vc, kv_lens, scale=scale)


def decode_via(fwd):
    """Decode built from a prefill implementation: T = 1 query at the end of
    a sequence of kv_len keys."""
    def dec(q, kc, vc, kv_lens, scale=None):
        B, Hq, D = q.shape
        o = np.zeros((B, Hq, D))
        lse = np.full((B, Hq), -np.inf)
        for b in range(B):
            L = int(kv_lens[b])
            if L == 0:
                continue
            ob, lb = fwd(q[b:b + 1, :, None, :], kc[b:b + 1, :, :L],
                         vc[b:b + 1, :, :L], causal=True, key_lens=None,
                         scale=scale)
            o[b], lse[b] = ob[0, :, 0], lb[0, :, 0]
        return o, lse
    return dec


# ------------------------------------------------------------------ helpers

def _rng(seed):
    return np.random.default_rng(seed)


def _expected_rows(T, S, L, causal):
    """For each query row: None if it has no visible key, else hi such that
    keys 0..hi-1 are the visible ones (bottom-right alignment)."""
    out = []
    for i in range(T):
        pos = i + S - T
        if pos >= L:
            out.append(None)
            continue
        hi = min(L, pos + 1) if causal else L
        out.append(hi if hi > 0 else None)
    return out


MASK_CASES = [
    # (T, S, causal, key_lens)
    (13, 13, True, None),
    (5, 13, True, None),        # T < S: bottom-right causal
    (13, 5, True, None),        # T > S: first rows see no key
    (13, 13, False, [13, 6]),   # key padding, padded query rows
    (13, 13, True, [13, 6]),    # causal + padding
    (7, 13, False, [9, 13]),    # non-causal, T < S, padding
    (13, 13, True, [0, 1]),     # empty and single-key sequences
]


# --------------------------------------------------------------------- pins

def pin_uniform_scores(fwd):
    """Q = 0: all visible scores are 0, so O[i] is the plain mean of the
    visible value rows and LSE[i] = ln(number of visible keys).  Pins the
    causal/padding masks, bottom-right alignment, padded rows, the GQA head
    mapping (each KV head has different values) and the LSE base."""
    rng = _rng(11)
    B, Hq, Hkv, D = 2, 4, 2, 6
    G = Hq // Hkv
    for T, S, causal, lens in MASK_CASES:
        q = np.zeros((B, Hq, T, D))
        k = rng.normal(size=(B, Hkv, S, D))
        v = rng.normal(size=(B, Hkv, S, D))
        o, lse = fwd(q, k, v, causal=causal, key_lens=lens, scale=0.37)
        for b in range(B):
            L = S if lens is None else lens[b]
            for h in range(Hq):
                g = h // G
                for i, hi in enumerate(_expected_rows(T, S, L, causal)):
                    if hi is None:
                        assert np.all(o[b, h, i] == 0.0), (T, S, b, h, i)
                        assert lse[b, h, i] == -np.inf, (T, S, b, h, i)
                    else:
                        want = v[b, g, :hi].mean(axis=0)
                        np.testing.assert_allclose(o[b, h, i], want, rtol=0, atol=ATOL)
                        assert abs(lse[b, h, i] - math.log(hi)) < ATOL


def pin_two_keys(fwd):
    """Two keys: the weight of key 0 is the logistic function of s0 - s1 and
    LSE = logaddexp(s0, s1), with s_j = scale * q . k_j.  Includes scores of
    several hundred, which overflow exp() without the max subtraction."""
    rng = _rng(12)
    D = 5
    for a, b0, b1, scale in [(1.0, 0.5, -0.25, 0.7), (3.0, -1.0, 2.0, 0.125),
                             (40.0, 30.0, 29.5, 0.9), (-25.0, 40.0, -40.0, 1.0)]:
        q = np.zeros((1, 1, 1, D)); q[..., 0] = a
        k = rng.normal(size=(1, 1, 2, D)); k[0, 0, 0, 0] = b0; k[0, 0, 1, 0] = b1
        q[..., 1:] = 0.0
        v = rng.normal(size=(1, 1, 2, D))
        o, lse = fwd(q, k, v, causal=False, key_lens=None, scale=scale)
        s0, s1 = scale * a * b0, scale * a * b1
        w0 = 1.0 / (1.0 + math.exp(s1 - s0)) if s1 - s0 < 700 else 0.0
        want = w0 * v[0, 0, 0] + (1.0 - w0) * v[0, 0, 1]
        np.testing.assert_allclose(o[0, 0, 0], want, rtol=0, atol=1e-12)
        assert abs(lse[0, 0, 0] - np.logaddexp(s0, s1)) < 1e-9 * max(1, abs(s0))


def pin_single_key(fwd):
    """One visible key: O = V[0], LSE = scale * q . k_0 (S = 1, and a padded
    batch whose valid length is 1)."""
    rng = _rng(13)
    D = 7
    q = rng.normal(size=(2, 3, 1, D))
    k = rng.normal(size=(2, 3, 1, D))
    v = rng.normal(size=(2, 3, 1, D))
    o, lse = fwd(q, k, v, causal=True, key_lens=None, scale=0.3)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=ATOL)
    np.testing.assert_allclose(lse[:, :, 0],
                               0.3 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]),
                               rtol=0, atol=ATOL)
    q = rng.normal(size=(1, 2, 4, D))
    k = rng.normal(size=(1, 2, 4, D))
    v = rng.normal(size=(1, 2, 4, D))
    o, _ = fwd(q, k, v, causal=False, key_lens=[1], scale=0.3)
    # S - T = 0, so only row 0 is a valid (non-padded) query row.
    np.testing.assert_allclose(o[0, :, 0], v[0, :, 0], rtol=0, atol=ATOL)
    assert np.all(o[0, :, 1:] == 0)


def pin_identical_values(fwd):
    """Every value row equal to c gives O = c on every row with a visible key."""
    rng = _rng(14)
    B, Hq, Hkv, T, S, D = 2, 4, 4, 9, 11, 5
    c = rng.normal(size=(B, Hkv, 1, D))
    v = np.broadcast_to(c, (B, Hkv, S, D)).copy()
    q = rng.normal(size=(B, Hq, T, D)) * 3
    k = rng.normal(size=(B, Hkv, S, D))
    o, _ = fwd(q, k, v, causal=True, key_lens=None, scale=0.5)
    np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0, atol=1e-12)


def pin_causal_row0(fwd):
    """Causal self-attention (T = S): row 0 sees only key 0, so O[0] = V[0]."""
    rng = _rng(15)
    q = rng.normal(size=(2, 2, 10, 4)) * 4
    k = rng.normal(size=(2, 2, 10, 4))
    v = rng.normal(size=(2, 2, 10, 4))
    o, _ = fwd(q, k, v, causal=True, key_lens=None, scale=0.5)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=ATOL)


def pin_weights_convex(fwd):
    """V = identity (D = S) makes O equal to the weight matrix.  Each row with
    a visible key is a convex combination: entries >= 0, exactly 0 on hidden
    keys, summing to 1; log-weight differences equal score differences; and
    LSE = s_j - ln w_j for every visible j."""
    rng = _rng(16)
    for T, S, causal, lens in MASK_CASES:
        B, Hq, Hkv = 2, 2, 1
        q = rng.normal(size=(B, Hq, T, S)) * 2
        k = rng.normal(size=(B, Hkv, S, S))
        v = np.broadcast_to(np.eye(S), (B, Hkv, S, S)).copy()
        scale = 0.6
        w, lse = fwd(q, k, v, causal=causal, key_lens=lens, scale=scale)
        for b in range(B):
            L = S if lens is None else lens[b]
            for h in range(Hq):
                for i, hi in enumerate(_expected_rows(T, S, L, causal)):
                    row = w[b, h, i]
                    if hi is None:
                        assert np.all(row == 0)
                        continue
                    assert np.all(row[hi:] == 0.0), (T, S, b, h, i)
                    assert np.all(row[:hi] > 0.0)
                    assert abs(row.sum() - 1.0) < 1e-12
                    s = scale * (k[b, 0, :hi] @ q[b, h, i])
                    np.testing.assert_allclose(np.log(row[:hi]) - np.log(row[0]),
                                               s - s[0], rtol=0, atol=1e-10)
                    np.testing.assert_allclose(s - np.log(row[:hi]),
                                               np.full(hi, lse[b, h, i]),
                                               rtol=0, atol=1e-10)


def pin_key_shift(fwd):
    """Adding the same vector u to every key shifts each row's scores by
    scale * q . u: O is unchanged and LSE moves by exactly that amount."""
    rng = _rng(17)
    B, Hq, Hkv, T, S, D = 1, 2, 2, 6, 9, 4
    q = rng.normal(size=(B, Hq, T, D))
    k = rng.normal(size=(B, Hkv, S, D))
    v = rng.normal(size=(B, Hkv, S, D))
    u = rng.normal(size=(D,))
    o1, l1 = fwd(q, k, v, causal=True, key_lens=None, scale=0.8)
    o2, l2 = fwd(q, k + u, v, causal=True, key_lens=None, scale=0.8)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2 - l1, 0.8 * (q @ u), rtol=0, atol=1e-12)


def pin_key_permutation(fwd):
    """Non-causal attention does not depend on the order of the (valid) keys."""
    rng = _rng(18)
    B, Hq, Hkv, T, S, D = 2, 2, 1, 5, 12, 4
    q = rng.normal(size=(B, Hq, T, D))
    k = rng.normal(size=(B, Hkv, S, D))
    v = rng.normal(size=(B, Hkv, S, D))
    lens = [12, 8]
    o1, l1 = fwd(q, k, v, causal=False, key_lens=lens, scale=0.4)
    k2, v2 = k.copy(), v.copy()
    for b, L in enumerate(lens):
        p = rng.permutation(L)
        k2[b, :, :L] = k[b][:, p]
        v2[b, :, :L] = v[b][:, p]
    o2, l2 = fwd(q, k2, v2, causal=False, key_lens=lens, scale=0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-12)


def pin_tiled_online(fwd):
    """The tiled online-softmax recurrence equals the full softmax (the
    method is exact: "FlashAttention", section 9.4.1)."""
    rng = _rng(19)
    B, Hq, Hkv, D = 1, 2, 1, 8
    for T, S, causal, lens in MASK_CASES[:5]:
        q = rng.normal(size=(B, Hq, T, D)) * 2
        k = rng.normal(size=(B, Hkv, S, D))
        v = rng.normal(size=(B, Hkv, S, D))
        L = None if lens is None else lens[:1]
        o, lse = fwd(q, k, v, causal=causal, key_lens=L, scale=0.35)
        for tq, tk in [(64, 64), (4, 3), (1, 1)]:
            ot, lt = oracle.attn_tiled_online_np(q, k, v, causal=causal,
                                                 key_lens=L, scale=0.35,
                                                 tile_q=tq, tile_k=tk)
            np.testing.assert_allclose(o, ot, rtol=0, atol=1e-12)
            np.testing.assert_array_equal(np.isinf(lse), np.isinf(lt))
            fin = np.isfinite(lse)
            np.testing.assert_allclose(lse[fin], lt[fin], rtol=0, atol=1e-12)


def pin_sdpa(fwd):
    """torch's float64 scaled_dot_product_attention with an explicit boolean
    mask (True = may attend), on rows that have a visible key."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = _rng(20)
    B, Hq, Hkv, D = 2, 4, 2, 8
    G = Hq // Hkv
    for T, S, causal, lens in MASK_CASES:
        q = rng.normal(size=(B, Hq, T, D))
        k = rng.normal(size=(B, Hkv, S, D))
        v = rng.normal(size=(B, Hkv, S, D))
        o, _ = fwd(q, k, v, causal=causal, key_lens=lens, scale=0.42)
        for b in range(B):
            L = S if lens is None else lens[b]
            rows = _expected_rows(T, S, L, causal)
            mask = np.zeros((T, S), dtype=bool)
            for i, hi in enumerate(rows):
                if hi is not None:
                    mask[i, :hi] = True
            good = np.array([hi is not None for hi in rows])
            if not good.any():
                continue
            kk = torch.from_numpy(np.repeat(k[b], G, axis=0))
            vv = torch.from_numpy(np.repeat(v[b], G, axis=0))
            ref = F.scaled_dot_product_attention(
                torch.from_numpy(q[b][:, good]), kk, vv,
                attn_mask=torch.from_numpy(mask[good]), scale=0.42).numpy()
            np.testing.assert_allclose(o[b][:, good], ref, rtol=0, atol=1e-12)


def pin_gqa_repeat(fwd):
    """Grouped-query attention equals multi-head attention with every KV head
    repeated for its group of Hq/Hkv consecutive query heads."""
    rng = _rng(21)
    B, Hq, Hkv, T, S, D = 2, 8, 2, 6, 7, 4
    q = rng.normal(size=(B, Hq, T, D))
    k = rng.normal(size=(B, Hkv, S, D))
    v = rng.normal(size=(B, Hkv, S, D))
    o1, l1 = fwd(q, k, v, causal=True, key_lens=[7, 5], scale=0.5)
    G = Hq // Hkv
    o2, l2 = fwd(q, np.repeat(k, G, axis=1), np.repeat(v, G, axis=1),
                 causal=True, key_lens=[7, 5], scale=0.5)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(l1, l2)


def pin_incremental_decode(fwd, dec):
    """Incremental decoding equals the full causal forward at every step:
    step t appends token t and its query sees cache rows 0..t
    ("Implementing attention from scratch", KV caching and Testing)."""
    rng = _rng(22)
    B, Hq, Hkv, n, D = 2, 4, 2, 9, 6
    q = rng.normal(size=(B, Hq, n, D)) * 2
    k = rng.normal(size=(B, Hkv, n, D))
    v = rng.normal(size=(B, Hkv, n, D))
    of, lf = fwd(q, k, v, causal=True, key_lens=None, scale=0.45)
    kc = np.zeros((B, Hkv, n + 3, D))
    vc = np.zeros((B, Hkv, n + 3, D))
    for t in range(n):
        # append token t at offset t (cache length before the append)
        oracle.kv_append(kc, vc, k[:, :, t], v[:, :, t], np.full(B, t))
        od, ld = dec(q[:, :, t], kc, vc, np.full(B, t + 1), scale=0.45)
        np.testing.assert_allclose(od, of[:, :, t], rtol=0, atol=1e-12)
        np.testing.assert_allclose(ld, lf[:, :, t], rtol=0, atol=1e-12)


PREFILL_PINS = [pin_uniform_scores, pin_two_keys, pin_single_key,
                pin_identical_values, pin_causal_row0, pin_weights_convex,
                pin_key_shift, pin_key_permutation, pin_tiled_online, pin_sdpa,
                pin_gqa_repeat]

IMPLS = {"c": (c_fwd, c_dec), "numpy": (np_fwd, np_dec)}


@pytest.mark.parametrize("impl", list(IMPLS))
@pytest.mark.parametrize("pin", PREFILL_PINS, ids=lambda p: p.__name__)
def test_prefill_pin(impl, pin):
    pin(IMPLS[impl][0])


@pytest.mark.parametrize("impl", list(IMPLS))
def test_incremental_decode_pin(impl):
    fwd, dec = IMPLS[impl]
    pin_incremental_decode(fwd, dec)


def test_c_and_numpy_agree_random():
    """The two independent implementations agree to float64 rounding on a
    random case with every feature switched on."""
    rng = _rng(23)
    q = rng.normal(size=(3, 6, 21, 16)) * 2
    k = rng.normal(size=(3, 2, 29, 16))
    v = rng.normal(size=(3, 2, 29, 16))
    for causal in (False, True):
        o1, l1 = c_fwd(q, k, v, causal=causal, key_lens=[29, 17, 3])
        o2, l2 = np_fwd(q, k, v, causal=causal, key_lens=[29, 17, 3])
        np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
        np.testing.assert_array_equal(np.isinf(l1), np.isinf(l2))
        fin = np.isfinite(l1)
        np.testing.assert_allclose(l1[fin], l2[fin], rtol=0, atol=1e-13)


def test_row_sampling_matches_full():
    """Sampled rows (used at full benchmark sizes) equal the same rows of a
    full run."""
    rng = _rng(24)
    q = rng.normal(size=(2, 4, 17, 8))
    k = rng.normal(size=(2, 2, 19, 8))
    v = rng.normal(size=(2, 2, 19, 8))
    o, l = c_fwd(q, k, v, causal=True, key_lens=[19, 11])
    rows = rng.choice(2 * 4 * 17, size=40, replace=False).astype(np.int64)
    os_, ls_ = oracle.attn_fwd(q, k, v, causal=True, key_lens=[19, 11],
                               rows=rows, nthreads=3)
    np.testing.assert_array_equal(os_, o.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(ls_, l.reshape(-1)[rows])


def test_bf16_widening_is_exact():
    """bf16 inputs are widened exactly: the oracle on raw bf16 bits equals the
    oracle on the float64 values torch assigns to the same bf16 numbers."""
    torch = pytest.importorskip("torch")
    g = torch.Generator().manual_seed(5)
    x = torch.randn(1, 2, 9, 8, generator=g).to(torch.bfloat16)
    y = torch.randn(1, 1, 11, 8, generator=g).to(torch.bfloat16)
    z = torch.randn(1, 1, 11, 8, generator=g).to(torch.bfloat16)
    bits = [t.view(torch.int16).numpy().view(np.uint16) for t in (x, y, z)]
    np.testing.assert_array_equal(oracle.bf16_bits_to_f64(bits[0]),
                                  x.double().numpy())
    o1, l1 = oracle.attn_fwd(*bits, causal=True, bf16=True)
    o2, l2 = oracle.attn_fwd(x.double().numpy(), y.double().numpy(),
                             z.double().numpy(), causal=True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_bad_arguments_rejected():
    q = np.zeros((1, 3, 4, 8))
    k = np.zeros((1, 2, 4, 8))
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, k)  # Hq % Hkv != 0
    q = np.zeros((1, 2, 4, 8))
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k, k, key_lens=[5])  # key_lens > S


def test_kv_cache_growth_golden():
    """Cache growth fixture: after 10 single-token appends the cache holds 10
    positions ("Building a causal self-attention block", Running and Testing
    It: (1, 4, 1, 16) grows to (1, 4, 10, 16)); appended rows are stored
    bit-for-bit and an out-of-range position is skipped."""
    with open(os.path.join(GOLDEN, "kv_cache_growth.json")) as f:
        fx = json.load(f)
    B, H, _, D = fx["shape_after_first_step"]
    steps = fx["steps"]
    assert fx["shape_after_last_step"] == [B, H, steps, D]
    rng = _rng(25)
    kc = np.full((B, H, steps, D), np.nan, dtype=np.float32)
    vc = np.full((B, H, steps, D), np.nan, dtype=np.float32)
    toks = rng.normal(size=(steps, 2, B, H, D)).astype(np.float32)
    for t in range(steps):
        assert oracle.kv_append(kc, vc, toks[t, 0], toks[t, 1], [t]) == 0
        filled = int(np.isfinite(kc[0, 0, :, 0]).sum())
        assert [B, H, filled, D] == ([B, H, 1, D] if t == 0 else [B, H, t + 1, D])
    np.testing.assert_array_equal(kc, np.moveaxis(toks[:, 0], 0, 2))
    np.testing.assert_array_equal(vc, np.moveaxis(toks[:, 1], 0, 2))
    assert oracle.kv_append(kc, vc, toks[0, 0], toks[0, 1], [steps]) == B * H


def test_page1_config_fixture():
    """The NumPy build guide's worked configuration (Step 1: n=256, m=512,
    d=64, T_q=T_k=64, seed 0) and its Verification claim that a correct tiled
    result is within 1e-5 of the naive one: on those exact float32 inputs the
    tiled online recurrence and the full definition, both in float64, agree
    far inside that bound."""
    with open(os.path.join(GOLDEN, "page1_config.json")) as f:
        fx = json.load(f)
    np.random.seed(fx["seed"])
    n, m, d = fx["n"], fx["m"], fx["d"]
    Q = np.random.randn(n, d).astype(np.float32)
    K = np.random.randn(m, d).astype(np.float32)
    V = np.random.randn(m, d).astype(np.float32)
    q, k, v = (x[None, None].astype(np.float64) for x in (Q, K, V))
    o, _ = c_fwd(q, k, v)
    ot, _ = oracle.attn_tiled_online_np(q, k, v, tile_q=fx["T_q"], tile_k=fx["T_k"])
    err = np.abs(o - ot).max()
    assert err < fx["claimed_max_abs_error_bound"]
    assert err < 1e-12


def test_page1_step5_reading():
    """Reading of the NumPy guide's Step 5: normalising each key tile on its
    own and adding the tiles is not softmax (each row's weights then sum to
    the number of key tiles), so it cannot be the oracle; the online
    recurrence is."""
    rng = _rng(26)
    n, m, d, tk = 8, 32, 4, 8
    q = rng.normal(size=(n, d))
    k = rng.normal(size=(m, d))
    ones = np.ones((m, 1))
    per_tile = np.zeros((n, 1))
    for k0 in range(0, m, tk):
        s = q @ k[k0:k0 + tk].T / math.sqrt(d)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        per_tile += (w / w.sum(axis=1, keepdims=True)) @ ones[k0:k0 + tk]
    np.testing.assert_allclose(per_tile, m // tk)
    o, _ = c_fwd(q[None, None], k[None, None], ones.repeat(d, 1)[None, None])
    np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-13)


# ------------------------------------------------------ planted mistakes

def _mutant(mistake):
    """A small CPU copy of the definition with one planted mistake."""
    def fwd(q, k, v, causal=False, key_lens=None, scale=None):
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        B, Hq, T, D = q.shape
        _, Hkv, S, _ = k.shape
        G = Hq // Hkv
        if scale is None or mistake == "default_scale":
            scale = 1.0 / math.sqrt(D)
        o = np.zeros((B, Hq, T, D))
        lse = np.full((B, Hq, T), -np.inf)
        with np.errstate(all="ignore"):
            for b in range(B):
                L = S if (key_lens is None or mistake == "ignore_lens") else int(key_lens[b])
                for h in range(Hq):
                    g = h % Hkv if mistake == "gqa_modulo" else h // G
                    s = q[b, h] @ k[b, g].T
                    if mistake != "no_scale":
                        s = s * scale
                    pos = np.arange(T)[:, None] + (0 if mistake == "topleft" else S - T)
                    j = np.arange(S)[None, :]
                    vis = np.broadcast_to(j < (L - 1 if mistake == "drop_last_key" else L),
                                          (T, S)).copy()
                    if causal:
                        vis &= (j < pos) if mistake == "offbyone" else (j <= pos)
                    valid = pos[:, 0] < L
                    if mistake != "keep_padded_rows":
                        vis &= valid[:, None]
                    s = np.where(vis, s, -np.inf)
                    ax = 0 if mistake == "softmax_axis0" else 1
                    m = s.max(axis=ax, keepdims=True)
                    if mistake == "no_max":
                        m = np.zeros_like(m)
                    if mistake != "nan_rows":
                        m = np.where(np.isfinite(m), m, 0.0)
                    e = np.exp((m - s) if mistake == "sign" else (s - m))
                    e = np.where(vis, e, 0.0) if mistake != "nan_rows" else np.exp(s - m)
                    if mistake == "tile_local":
                        w = np.zeros_like(e)
                        for k0 in range(0, S, 4):
                            blk = e[:, k0:k0 + 4]
                            zz = blk.sum(axis=1, keepdims=True)
                            w[:, k0:k0 + 4] = np.where(zz > 0, blk / np.where(zz > 0, zz, 1), 0)
                    else:
                        z = e.sum(axis=ax, keepdims=True)
                        w = e if mistake == "no_norm" else np.where(z > 0, e / np.where(z > 0, z, 1), 0)
                    vals = k[b, g] if mistake == "k_for_v" else v[b, g]
                    if mistake == "v_roll":
                        vals = np.roll(vals, 1, axis=0)
                    o[b, h] = w @ vals
                    zr = e.sum(axis=1)
                    mr = m[:, 0] if ax == 1 else s.max(axis=1)
                    if mistake == "lse_no_max":
                        l = np.log(zr)
                    elif mistake == "lse_log2":
                        l = (mr + np.log(zr)) / math.log(2)
                    else:
                        l = mr + np.log(zr)
                    has = vis.any(axis=1) if mistake != "nan_rows" else np.ones(T, bool)
                    lse[b, h] = np.where(has, l, -np.inf)
        return o, lse
    return fwd


MISTAKES = ["no_scale", "default_scale", "topleft", "offbyone", "drop_last_key",
            "ignore_lens", "keep_padded_rows", "gqa_modulo", "softmax_axis0",
            "no_max", "sign", "no_norm", "nan_rows", "tile_local", "k_for_v",
            "v_roll", "lse_no_max", "lse_log2"]


def _fails_some_pin(fwd):
    dec = decode_via(fwd)
    for pin in PREFILL_PINS:
        try:
            pin(fwd)
        except (AssertionError, FloatingPointError):
            return pin.__name__
    try:
        pin_incremental_decode(fwd, dec)
    except (AssertionError, FloatingPointError):
        return "pin_incremental_decode"
    return None


def test_clean_copy_passes_all_pins():
    assert _fails_some_pin(_mutant(None)) is None


@pytest.mark.parametrize("mistake", MISTAKES)
def test_pins_catch_planted_mistakes(mistake):
    caught_by = _fails_some_pin(_mutant(mistake))
    assert caught_by is not None, f"no pin catches the planted mistake {mistake!r}"


def test_f16_inputs_are_widened_exactly():
    """fp16 inputs reach the oracle as their exact float64 values: the C
    oracle on float16 arrays equals the C oracle on the same values stored
    as float64, and both equal the NumPy twin."""
    r = _rng(77)
    q, k, v = (r.standard_normal(s).astype(np.float16) for s in
               ((2, 2, 9, 8), (2, 1, 11, 8), (2, 1, 11, 8)))
    a = oracle.attn_fwd(q, k, v, causal=True, nthreads=1)
    b = oracle.attn_fwd(q.astype(np.float64), k.astype(np.float64), v.astype(np.float64),
                        causal=True, nthreads=1)
    c = oracle.attn_fwd_np(q, k, v, causal=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.allclose(a[0], c[0], atol=ATOL) and np.allclose(a[1], c[1], atol=ATOL)
    # every float16 value is a float64 value exactly (11-bit significand)
    x = np.arange(-65504, 65505, 97, dtype=np.float64).astype(np.float16)
    assert np.array_equal(x.astype(np.float64).astype(np.float16), x)
