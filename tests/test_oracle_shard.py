"""Pins for the oracle's key-shard attention and LSE merge (CPU only).

"Building a causal self-attention block from scratch in PyTorch", Extending
It: distributed attention shards Q/K/V across devices and recombines the
results.  oracle.attn_fwd_kv_shard_np computes the attention of the queries
over one shard of the keys (global positions), oracle.lse_merge_np combines
partials over disjoint key sets.  Neither is re-typed here; they are pinned
to what the mathematics fixes:

* any split of the keys into shards, merged, is the full attention of the
  C oracle (already pinned to the definition) -- for causal, non-causal,
  key padding, T < S, chunked query positions and GQA;
* one shard holding every key is attn_fwd_np with the same query positions;
* Q = 0 gives every shard the mean of its visible value rows and LSE = ln
  of their count;
* the merge is the identity on one partial, ignores partials with LSE =
  -inf, does not depend on the order of the partials, follows the two-part
  closed form O = (Z1 O1 + Z2 O2) / (Z1 + Z2), and does not overflow for
  large LSE;
* planted mistakes in small copies (the shard offset ignored, rows padded
  by the shard's own length, a merge without weights, without its maximum,
  or returning the largest LSE) each fail a pin.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

CASES = [
    # (B, Hq, Hkv, T, S_full, D, causal, key_lens, q_pos)
    (2, 2, 1, 7, 13, 4, True, [13, 9], [6, 2]),      # bottom-right-ish, padding, GQA
    (1, 2, 2, 5, 11, 3, False, [8], [0]),            # non-causal with padding
    (2, 1, 1, 9, 9, 5, True, [9, 5], [0, 0]),        # self-attention, padded rows
    (1, 4, 2, 4, 16, 4, True, [16], [12]),           # decode-like chunk at the end
]


def _inputs(case, seed):
    B, Hq, Hkv, T, S, D = case[:6]
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, Hq, T, D)), r.standard_normal((B, Hkv, S, D)),
            r.standard_normal((B, Hkv, S, D)))


def _splits(S, rng, n):
    cuts = np.sort(rng.choice(np.arange(1, S), size=min(n - 1, S - 1), replace=False))
    return [0, *cuts.tolist(), S]


def pin_shards_merge_to_full(shard_fn, merge_fn, case, seed=1):
    q, k, v = _inputs(case, seed)
    B, Hq, Hkv, T, S, D, causal, lens, qp = case
    lens, qp = np.array(lens, np.int32), np.array(qp, np.int32)
    ref_o, ref_l = oracle.attn_fwd(q, k, v, causal=causal, key_lens=lens, q_pos=qp, nthreads=1)
    rng = np.random.default_rng(seed + 10)
    for n in (1, 2, 3, 5):
        cut = _splits(S, rng, n)
        parts = [shard_fn(q, k[:, :, a:b], v[:, :, a:b], qp, lens, a, causal=causal)
                 for a, b in zip(cut[:-1], cut[1:])]
        o, lse = merge_fn(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
        assert np.allclose(o, ref_o, atol=1e-12), f"{n} shards"
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(lse), fin)
        assert np.allclose(lse[fin], ref_l[fin], atol=1e-12)
        assert np.all(o[~fin] == 0)


def pin_one_shard_is_chunked_prefill(shard_fn, merge_fn, case, seed=2):
    q, k, v = _inputs(case, seed)
    causal, lens, qp = case[6], np.array(case[7], np.int32), np.array(case[8], np.int32)
    o, lse = shard_fn(q, k, v, qp, lens, 0, causal=causal)
    ro, rl = oracle.attn_fwd_np(q, k, v, causal=causal, key_lens=lens, q_pos=qp)
    assert np.allclose(o, ro, atol=1e-12)
    assert np.array_equal(np.isneginf(lse), np.isneginf(rl))


def pin_zero_queries(shard_fn, merge_fn, case, seed=3):
    """Q = 0: the shard's weights are uniform over its visible keys."""
    q, k, v = _inputs(case, seed)
    B, Hq, Hkv, T, S, D, causal, lens, qp = case
    G = Hq // Hkv
    a, b = S // 3, S // 3 + max(1, S // 2)
    o, lse = shard_fn(np.zeros_like(q), k[:, :, a:b], v[:, :, a:b], np.array(qp, np.int32),
                      np.array(lens, np.int32), a, causal=causal)
    for bb in range(B):
        for h in range(Hq):
            for i in range(T):
                p = qp[bb] + i
                xs = [x for x in range(a, b) if x < lens[bb] and p < lens[bb]
                      and (not causal or x <= p)]
                if not xs:
                    assert np.all(o[bb, h, i] == 0) and np.isneginf(lse[bb, h, i])
                    continue
                want = v[bb, h // G, xs].mean(axis=0)
                assert np.allclose(o[bb, h, i], want, atol=1e-12)
                assert abs(lse[bb, h, i] - np.log(len(xs))) <= 1e-12


def pin_merge_identities(shard_fn, merge_fn, case=None, seed=4):
    r = np.random.default_rng(seed)
    o1, o2 = r.standard_normal((2, 3, 5, 4))
    l1, l2 = r.standard_normal((2, 3, 5)) * 3
    # one part: identity
    o, lse = merge_fn(o1[None], l1[None])
    assert np.allclose(o, o1, atol=1e-14) and np.allclose(lse, l1, atol=1e-14)
    # a part that saw nothing changes nothing
    o, lse = merge_fn(np.stack([o1, np.zeros_like(o1)]), np.stack([l1, np.full_like(l1, -np.inf)]))
    assert np.allclose(o, o1, atol=1e-14) and np.allclose(lse, l1, atol=1e-14)
    # two parts: closed form, and the order does not matter
    z1, z2 = np.exp(l1), np.exp(l2)
    want = (z1[..., None] * o1 + z2[..., None] * o2) / (z1 + z2)[..., None]
    for parts in ((o1, o2, l1, l2), (o2, o1, l2, l1)):
        o, lse = merge_fn(np.stack(parts[:2]), np.stack(parts[2:]))
        assert np.allclose(o, want, atol=1e-12)
        assert np.allclose(lse, np.log(z1 + z2), atol=1e-12)
    # large LSE: no overflow (the result only depends on the differences)
    o, lse = merge_fn(np.stack([o1, o2]), np.stack([l1 + 900.0, l2 + 900.0]))
    assert np.allclose(o, want, atol=1e-12) and np.allclose(lse, np.log(z1 + z2) + 900.0)
    # no part saw anything: O = 0, LSE = -inf
    o, lse = merge_fn(np.stack([o1, o2]), np.full((2, 3, 5), -np.inf))
    assert np.all(o == 0) and np.all(np.isneginf(lse))


PINS = [pin_shards_merge_to_full, pin_one_shard_is_chunked_prefill, pin_zero_queries,
        pin_merge_identities]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + f"-c{int(c[6])}")
@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_shard_pin(pin, case):
    pin(oracle.attn_fwd_kv_shard_np, oracle.lse_merge_np, case)


# ------------------------------------------------------- planted mistakes

def _small_shard(mistake=None):
    def fn(q, k, v, q_pos, key_lens, k_off, causal=True):
        B, Hq, T, D = q.shape
        _, Hkv, S, _ = k.shape
        G = Hq // Hkv
        o, lse = np.zeros((B, Hq, T, D)), np.full((B, Hq, T), -np.inf)
        off = 0 if mistake == "no_offset" else k_off
        for b in range(B):
            L = int(key_lens[b])
            for h in range(Hq):
                for i in range(T):
                    p = int(q_pos[b]) + i
                    pad = (p - off >= min(max(L - off, 0), S)) if mistake == "local_padding" \
                        else p >= L
                    js = [j for j in range(S) if off + j < L and not pad
                          and (not causal or off + j <= p)]
                    if not js:
                        continue
                    s = k[b, h // G, js] @ q[b, h, i] / np.sqrt(D)
                    e = np.exp(s - s.max())
                    o[b, h, i] = e @ v[b, h // G, js] / e.sum()
                    lse[b, h, i] = s.max() + np.log(e.sum())
        return o, lse
    return fn


def _small_merge(mistake=None):
    def fn(o_parts, lse_parts):
        fin = np.isfinite(lse_parts)
        m = np.where(fin, lse_parts, -np.inf).max(axis=0)
        has = np.isfinite(m)
        ref = np.where(has, m, 0.0) if mistake != "no_max" else np.zeros_like(m)
        w = np.where(fin, np.exp(np.where(fin, lse_parts, 0.0) - ref), 0.0)
        if mistake == "unweighted":
            w = fin.astype(float)
        z = np.where(has, w.sum(axis=0), 1.0)
        o = np.where(has[..., None], (w[..., None] * o_parts).sum(axis=0) / z[..., None], 0.0)
        lse = np.where(has, ref + np.log(z), -np.inf)
        if mistake == "lse_max":
            lse = np.where(has, m, -np.inf)
        return o, lse
    return fn


def test_clean_small_copies_pass_pins():
    for case in CASES[:2]:
        for pin in PINS:
            pin(_small_shard(), _small_merge(), case)


@pytest.mark.parametrize("mistake", ["no_offset", "local_padding", "unweighted", "no_max",
                                     "lse_max"])
def test_pins_catch_planted_mistakes(mistake):
    shard = _small_shard(mistake if mistake in ("no_offset", "local_padding") else None)
    merge = _small_merge(mistake if mistake not in ("no_offset", "local_padding") else None)
    failed = 0
    for case in CASES[:2]:
        for pin in PINS:
            try:
                with np.errstate(all="ignore"):
                    pin(shard, merge, case)
            except AssertionError:
                failed += 1
    assert failed >= 1, f"no pin noticed {mistake}"
