"""Pins for the float64 attention backward in the oracle (CPU only).

The backward is the chain rule through the softmax ("Hands-on build guide:
FlashAttention-style tiled attention kernel in pure NumPy", Roadmap:
gradient through attention; "Implementing attention from scratch", Testing
against a reference: compare gradients with a float64 reference).  None of
the pins re-types it:

* finite differences: central differences of the oracle's own forward (the
  C implementation) on the loss <O, dO> match the analytic gradients;
* a library special case: torch float64 autograd through
  scaled_dot_product_attention with an explicit boolean mask;
* invariants: each row of dS sums to zero, so the key gradients of a (b,
  kv head) sum to zero and dQ does not change when every key moves by the
  same vector; the value gradients sum to the sum of dO over rows that see
  a key; keys nobody sees and rows that see nothing get zero gradients;
* planted mistakes in a small copy each fail a pin.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

CASES = [
    # (B, Hq, Hkv, T, S, D, causal, key_lens, q_pos)
    (2, 4, 2, 7, 7, 5, True, None, None),
    (2, 2, 1, 5, 9, 4, True, [9, 6], None),          # T < S, bottom-right, padding
    (1, 2, 2, 9, 5, 3, True, None, None),            # T > S: first rows see nothing
    (2, 2, 2, 6, 8, 4, False, [8, 3], None),
    (2, 4, 2, 4, 12, 6, True, [10, 12], [3, 8]),     # chunked: query positions q_pos
]


def _inputs(case, seed):
    B, Hq, Hkv, T, S, D = case[:6]
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, Hq, T, D)), r.standard_normal((B, Hkv, S, D)),
            r.standard_normal((B, Hkv, S, D)), r.standard_normal((B, Hq, T, D)))


def _kw(case):
    causal, lens, qp = case[6], case[7], case[8]
    return dict(causal=causal, key_lens=None if lens is None else np.array(lens, np.int32),
                q_pos=None if qp is None else np.array(qp, np.int32))


def bwd(q, k, v, do, **kw):
    dq, dk, dv, _, _ = oracle.attn_bwd_np(q, k, v, do, **kw)
    return dq, dk, dv


def pin_finite_differences(bwd_fn, case, seed=1):
    q, k, v, do = _inputs(case, seed)
    kw = _kw(case)
    dq, dk, dv = bwd_fn(q, k, v, do, **kw)

    def loss(qq, kk, vv):
        o, _ = oracle.attn_fwd(qq, kk, vv, nthreads=1, **kw)
        return float((o * do).sum())

    r = np.random.default_rng(seed + 100)
    eps = 1e-5
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(r.integers(0, n)) for n in x.shape)
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-7 * max(1.0, abs(fd)), (name, idx, fd, g[idx])


def pin_invariants(bwd_fn, case, seed=2):
    q, k, v, do = _inputs(case, seed)
    kw = _kw(case)
    B, Hq, Hkv, T, S, D = case[:6]
    G = Hq // Hkv
    dq, dk, dv = bwd_fn(q, k, v, do, **kw)
    # each row of dS sums to zero -> key gradients sum to zero per (b, g)
    assert np.allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    # value gradients sum to the sum of dO over rows that see a key
    for b in range(B):
        L = S if kw["key_lens"] is None else int(kw["key_lens"][b])
        qp = None if kw["q_pos"] is None else int(kw["q_pos"][b])
        _, vis = oracle.visibility(T, S, L, kw["causal"], qp)
        has = vis.any(axis=1)
        seen = vis.any(axis=0)
        for g in range(Hkv):
            want = sum(do[b, h][has].sum(axis=0) for h in range(g * G, (g + 1) * G))
            assert np.allclose(dv[b, g].sum(axis=0), want, atol=1e-12)
            assert np.all(dk[b, g][~seen] == 0) and np.all(dv[b, g][~seen] == 0)
        for h in range(Hq):
            assert np.all(dq[b, h][~has] == 0)
    # moving every key by the same vector leaves dQ unchanged
    u = np.random.default_rng(seed + 7).standard_normal(D)
    dq2, _, _ = bwd_fn(q, k + u, v, do, **kw)
    assert np.allclose(dq2, dq, atol=1e-10)


def pin_torch_autograd(bwd_fn, case, seed=3):
    torch = pytest.importorskip("torch")
    q, k, v, do = _inputs(case, seed)
    kw = _kw(case)
    B, Hq, Hkv, T, S, D = case[:6]
    G = Hq // Hkv
    mask = np.zeros((B, 1, T, S), bool)
    has = np.zeros((B, T), bool)
    for b in range(B):
        L = S if kw["key_lens"] is None else int(kw["key_lens"][b])
        qp = None if kw["q_pos"] is None else int(kw["q_pos"][b])
        _, vis = oracle.visibility(T, S, L, kw["causal"], qp)
        mask[b, 0] = vis
        has[b] = vis.any(axis=1)
    # rows that see no key are NaN in SDPA: give them one key and no gradient
    m_t = torch.from_numpy(mask | ~has[:, None, :, None])
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    kk = tk.repeat_interleave(G, dim=1)
    vv = tv.repeat_interleave(G, dim=1)
    o = torch.nn.functional.scaled_dot_product_attention(tq, kk, vv, attn_mask=m_t,
                                                         scale=1.0 / np.sqrt(D))
    dot = torch.from_numpy(do * has[:, None, :, None])
    (o * dot).sum().backward()
    dq, dk, dv = bwd_fn(q, k, v, do * has[:, None, :, None], **kw)
    assert np.allclose(tq.grad.numpy(), dq, atol=1e-10)
    assert np.allclose(tk.grad.numpy(), dk, atol=1e-10)
    assert np.allclose(tv.grad.numpy(), dv, atol=1e-10)


PINS = [pin_finite_differences, pin_invariants, pin_torch_autograd]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + f"-c{int(c[6])}")
@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_bwd_pin(pin, case):
    pin(bwd, case)


# ------------------------------------------------------- planted mistakes

def _small_bwd(mistake=None):
    """A small, separate copy of the backward for the planted-mistake check."""
    def fn(q, k, v, do, causal=False, key_lens=None, q_pos=None):
        B, Hq, T, D = q.shape
        _, Hkv, S, _ = k.shape
        G = Hq // Hkv
        sc = 1 / np.sqrt(D)
        dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for b in range(B):
            L = S if key_lens is None else int(key_lens[b])
            qp = None if q_pos is None else int(q_pos[b])
            _, vis = oracle.visibility(T, S, L, causal, qp)
            has = vis.any(axis=1)
            for h in range(Hq):
                g = h // G
                s = np.where(vis, sc * q[b, h] @ k[b, g].T, -np.inf)
                m = np.where(has, s.max(axis=1), 0)
                e = np.where(vis, np.exp(s - m[:, None]), 0)
                p = e / np.where(has, e.sum(axis=1), 1)[:, None]
                o = p @ v[b, g]
                dpv = p.T @ (o if mistake == "dv_from_o" else do[b, h])
                if mistake == "gqa_overwrite":
                    dv[b, g] = dpv
                else:
                    dv[b, g] += dpv
                dp = do[b, h] @ v[b, g].T
                delta = (do[b, h] * o).sum(axis=1)
                if mistake == "no_delta":
                    delta = 0 * delta
                ds = p * (dp - delta[:, None])
                dq[b, h] = (1 if mistake == "dq_unscaled" else sc) * ds @ k[b, g]
                dk[b, g] += (1 if mistake == "dk_unscaled" else sc) * ds.T @ q[b, h]
        return dq, dk, dv
    return fn


def test_clean_small_copy_passes_pins():
    for case in CASES[:2]:
        for pin in PINS:
            pin(_small_bwd(), case)


@pytest.mark.parametrize("mistake", ["dv_from_o", "gqa_overwrite", "no_delta", "dq_unscaled",
                                     "dk_unscaled"])
def test_pins_catch_planted_mistakes(mistake):
    failed = 0
    for case in CASES[:2]:
        for pin in PINS:
            try:
                pin(_small_bwd(mistake), case)
            except AssertionError:
                failed += 1
    assert failed >= 1, f"no pin noticed {mistake}"
