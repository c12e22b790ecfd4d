"""Pins for chunked prefill against a KV cache in the float64 oracle (CPU).

"Implementing attention from scratch", KV caching: a query that follows
``c`` cached tokens sits at key position ``c`` plus its position within the
chunk, and with a causal mask it sees every cached key and the chunk's keys
up to itself.  The oracle takes this as ``q_pos[b]`` (key position of query
row 0 of sequence b) and ``key_lens[b]`` (valid keys: cache + chunk).

Pins, none of which re-types the definition:

* chunked == full: running a sequence through ragged chunks against its
  growing cache reproduces the rows of one causal pass over the whole
  sequence ("Implementing attention from scratch", Testing against a
  reference: incremental results must match the full forward).  Cache rows
  past the valid length are NaN, so reading one would show.
* closed form: with Q = 0 every visible score is equal, so each row is the
  mean of the value rows 0..min(L, q_pos+i+1)-1 and LSE = ln(count); rows at
  or past L are padded (O = 0, LSE = -inf).
* the default: q_pos = S - T is exactly the bottom-right prefill.
* planted mistakes in a small copy (q_pos ignored, off by one, cache length
  ignored, q_pos taken as the chunk's end) each fail a pin.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

ATOL = 1e-12


def c_fwd(q, k, v, causal=True, key_lens=None, q_pos=None, scale=None):
    return oracle.attn_fwd(q, k, v, causal=causal, key_lens=key_lens, q_pos=q_pos,
                           scale=scale, nthreads=2)


def np_fwd(q, k, v, causal=True, key_lens=None, q_pos=None, scale=None):
    return oracle.attn_fwd_np(q, k, v, causal=causal, key_lens=key_lens, q_pos=q_pos,
                              scale=scale)


def _seq(seed, B=2, Hq=4, Hkv=2, N=23, D=8):
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, Hq, N, D)), r.standard_normal((B, Hkv, N, D)),
            r.standard_normal((B, Hkv, N, D)))


def pin_chunked_equals_full(fwd):
    """Per sequence, ragged chunk boundaries; the cache holds the first c + t
    rows of K/V and NaN beyond them."""
    Q, K, V = _seq(1)
    B, Hq, N, D = Q.shape
    S_max = N + 5
    full_o, full_l = oracle.attn_fwd_np(Q, K, V, causal=True)
    bounds = [[0, 1, 6, 7, 15, 23], [0, 9, 10, 17, 23]]   # chunk starts per sequence
    T = max(max(b[i + 1] - b[i] for i in range(len(b) - 1)) for b in bounds)
    steps = max(len(b) - 1 for b in bounds)
    for s in range(steps):
        q = np.zeros((B, Hq, T, D))
        kc = np.full((B, K.shape[1], S_max, D), np.nan)
        vc = np.full_like(kc, np.nan)
        q_pos = np.zeros(B, np.int32)
        lens = np.zeros(B, np.int32)
        for b in range(B):
            bb = bounds[b]
            if s >= len(bb) - 1:   # this sequence is done: an empty chunk
                c, t = bb[-1], 0
            else:
                c, t = bb[s], bb[s + 1] - bb[s]
            q[b, :, :t] = Q[b, :, c:c + t]
            kc[b, :, :c + t] = K[b, :, :c + t]
            vc[b, :, :c + t] = V[b, :, :c + t]
            q_pos[b], lens[b] = c, c + t
        o, l = fwd(q, kc, vc, causal=True, key_lens=lens, q_pos=q_pos)
        for b in range(B):
            c, t = int(q_pos[b]), int(lens[b] - q_pos[b])
            assert np.allclose(o[b, :, :t], full_o[b, :, c:c + t], atol=ATOL, rtol=0)
            assert np.allclose(l[b, :, :t], full_l[b, :, c:c + t], atol=ATOL, rtol=0)
            assert np.all(o[b, :, t:] == 0) and np.all(np.isneginf(l[b, :, t:]))


def pin_uniform_scores(fwd):
    """Q = 0: row i of sequence b is the mean of V rows 0..hi-1 with
    hi = min(L, q_pos + i + 1) (causal) or L (non-causal); LSE = ln hi."""
    r = np.random.default_rng(2)
    B, Hq, Hkv, T, S, D = 3, 4, 2, 6, 17, 5
    q = np.zeros((B, Hq, T, D))
    k = r.standard_normal((B, Hkv, S, D))
    v = r.standard_normal((B, Hkv, S, D))
    q_pos = np.array([0, 9, 14], np.int32)
    lens = np.array([4, 15, 17], np.int32)        # rows 4.., 6.., 3.. of the three are padded
    for causal in (True, False):
        o, l = fwd(q, k, v, causal=causal, key_lens=lens, q_pos=q_pos)
        for b in range(B):
            for h in range(Hq):
                g = h // (Hq // Hkv)
                for i in range(T):
                    pos = int(q_pos[b]) + i
                    if pos >= lens[b]:
                        assert np.all(o[b, h, i] == 0) and np.isneginf(l[b, h, i])
                        continue
                    hi = min(int(lens[b]), pos + 1) if causal else int(lens[b])
                    assert np.allclose(o[b, h, i], v[b, g, :hi].mean(axis=0), atol=ATOL)
                    assert abs(l[b, h, i] - np.log(hi)) <= ATOL


def pin_default_is_bottom_right(fwd):
    """q_pos = S - T for every sequence is the plain prefill."""
    r = np.random.default_rng(3)
    q = r.standard_normal((2, 2, 5, 4))
    k = r.standard_normal((2, 2, 9, 4))
    v = r.standard_normal((2, 2, 9, 4))
    lens = np.array([9, 6], np.int32)
    a = fwd(q, k, v, causal=True, key_lens=lens, q_pos=None)
    b = fwd(q, k, v, causal=True, key_lens=lens, q_pos=np.full(2, 4, np.int32))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


PINS = [pin_chunked_equals_full, pin_uniform_scores, pin_default_is_bottom_right]


@pytest.mark.parametrize("fwd", [c_fwd, np_fwd], ids=["c", "numpy"])
@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_chunked_pin(fwd, pin):
    pin(fwd)


def test_c_and_numpy_agree_on_chunks():
    r = np.random.default_rng(4)
    q = r.standard_normal((3, 4, 7, 16))
    k = r.standard_normal((3, 2, 30, 16))
    v = r.standard_normal((3, 2, 30, 16))
    q_pos = np.array([0, 11, 23], np.int32)
    lens = np.array([7, 15, 30], np.int32)
    for causal in (True, False):
        a = c_fwd(q, k, v, causal=causal, key_lens=lens, q_pos=q_pos)
        b = np_fwd(q, k, v, causal=causal, key_lens=lens, q_pos=q_pos)
        assert np.allclose(a[0], b[0], atol=ATOL) and np.array_equal(np.isneginf(a[1]),
                                                                     np.isneginf(b[1]))
        fin = np.isfinite(a[1])
        assert np.allclose(a[1][fin], b[1][fin], atol=ATOL)


# ------------------------------------------------------- planted mistakes

def _small_ref(mistake=None):
    """A small, separate copy of chunked attention used only to check that
    the pins notice plausible mistakes."""
    def fwd(q, k, v, causal=True, key_lens=None, q_pos=None, scale=None):
        B, Hq, T, D = q.shape
        _, Hkv, S, _ = k.shape
        scale = 1 / np.sqrt(D) if scale is None else scale
        o = np.zeros((B, Hq, T, D))
        lse = np.full((B, Hq, T), -np.inf)
        for b in range(B):
            L = S if key_lens is None else int(key_lens[b])
            c = S - T if q_pos is None else int(q_pos[b])
            if mistake == "ignore_q_pos":
                c = S - T
            if mistake == "q_pos_is_chunk_end":
                c = c - T
            if mistake == "ignore_lens":
                L = S
            for h in range(Hq):
                g = h // (Hq // Hkv)
                for i in range(T):
                    pos = c + i + (1 if mistake == "off_by_one" else 0)
                    if pos >= L:
                        continue
                    hi = min(L, pos + 1) if causal else L
                    if hi <= 0:
                        continue
                    s = scale * (k[b, g, :hi] @ q[b, h, i])
                    m = s.max()
                    w = np.exp(s - m)
                    o[b, h, i] = (w / w.sum()) @ v[b, g, :hi]
                    lse[b, h, i] = m + np.log(w.sum())
        return o, lse
    return fwd


def test_clean_small_copy_passes():
    for pin in PINS:
        pin(_small_ref())


@pytest.mark.parametrize("mistake", ["ignore_q_pos", "off_by_one", "ignore_lens",
                                     "q_pos_is_chunk_end"])
def test_pins_catch_planted_mistakes(mistake):
    failed = 0
    for pin in PINS:
        try:
            with np.errstate(invalid="ignore"):
                pin(_small_ref(mistake))
        except AssertionError:
            failed += 1
    assert failed >= 1, f"no pin noticed {mistake}"
