"""Pin of the backward's tolerance magnitudes (oracle.attn_bwd_magnitudes_np).

The GPU backward's elementwise bound is a small multiple of u * A, with u
the unit roundoff of one rounding (2^-8 for bf16) and A from
oracle.attn_bwd_magnitudes_np.  That function claims:
a backward that rounds P (for dV = P^T dO) and dS (for dQ and dK) to bf16,
forms delta = rowsum(dO * O) from the bf16-rounded O and rounds each result
once has, to first order, an error of at most u * A elementwise.

The claim is checked here without re-typing A's formula.  An evaluation of
the backward in float64 is written out below (independently of the oracle's
own backward), with a relative perturbation eps (|eps| <= u) applied at each
of those rounding points:

    O~  = O (1 + eps_O)               delta~ = rowsum(dO * O~)
    P~  = P (1 + eps_P)               dV~    = (sum_h P~^T dO) (1 + eps_dV)
    dS~ = P (dP - delta~) (1 + eps_S) dQ~    = scale dS~ K (1 + eps_dQ)
                                      dK~    = (sum_h scale dS~^T Q) (1 + eps_dK)

* random roundings: many draws of eps uniform in [-u, u] never move an
  element by more than u * A;
* worst-case roundings: for sampled elements, eps is aligned in sign with
  every term that reaches that element (the largest first-order change
  a rounding of at most u anywhere can cause); the change stays within
  u * A (up to second-order terms), and reaches most of it, so A is not
  a vacuous over-estimate;
* planted mistakes in a small copy of the magnitude formula (a dropped
  delta term, a dropped result rounding, P in place of |dS|, a dropped
  P^T |dO| term, a doubled bound) each fail one of these checks.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle

U = 2.0 ** -8   # bf16 unit roundoff

CASES = [
    # (B, Hq, Hkv, T, S, D, causal, key_lens, q_pos)
    (1, 2, 1, 9, 11, 5, True, None, None),             # GQA, bottom-right causal
    (2, 2, 2, 7, 7, 4, True, [7, 4], None),            # padding (padded rows)
    (1, 1, 1, 6, 9, 6, False, [7], None),              # non-causal with padding
    (2, 2, 1, 4, 10, 3, True, [9, 10], [3, 5]),        # chunked query positions
]


def _inputs(case, seed):
    B, Hq, Hkv, T, S, D = case[:6]
    r = np.random.default_rng(seed)
    return (r.standard_normal((B, Hq, T, D)), r.standard_normal((B, Hkv, S, D)),
            r.standard_normal((B, Hkv, S, D)), r.standard_normal((B, Hq, T, D)))


def _kw(case):
    lens, qp = case[7], case[8]
    return dict(causal=case[6], key_lens=None if lens is None else np.array(lens, np.int32),
                q_pos=None if qp is None else np.array(qp, np.int32))


def _vis(case, b, kw):
    T, S = case[3], case[4]
    L = S if kw["key_lens"] is None else int(kw["key_lens"][b])
    qp = None if kw["q_pos"] is None else int(kw["q_pos"][b])
    return oracle.visibility(T, S, L, kw["causal"], qp)[1]


def _softmax_rows(s, vis):
    """Row softmax over the visible entries (all-zero rows where none is)."""
    has = vis.any(axis=1)
    sm = np.where(vis, s, -np.inf)
    m = np.where(has, sm.max(axis=1), 0.0)
    e = np.where(vis, np.exp(sm - m[:, None]), 0.0)
    return e / np.where(has, e.sum(axis=1), 1.0)[:, None]


def zero_eps(case):
    B, Hq, Hkv, T, S, D = case[:6]
    return {"O": np.zeros((B, Hq, T, D)), "P": np.zeros((B, Hq, T, S)),
            "S": np.zeros((B, Hq, T, S)), "dQ": np.zeros((B, Hq, T, D)),
            "dK": np.zeros((B, Hkv, S, D)), "dV": np.zeros((B, Hkv, S, D))}


def intermediates(case, x):
    """P, O, dP and dS of every (b, h) in float64, unperturbed."""
    q, k, v, do = x
    kw = _kw(case)
    B, Hq, Hkv, T, S, D = case[:6]
    G, sc = Hq // Hkv, 1.0 / np.sqrt(D)
    out = {n: np.zeros((B, Hq, T, S)) for n in ("P", "dP", "dS")}
    out["O"] = np.zeros((B, Hq, T, D))
    for b in range(B):
        vis = _vis(case, b, kw)
        for h in range(Hq):
            g = h // G
            p = _softmax_rows(sc * q[b, h] @ k[b, g].T, vis)
            o = p @ v[b, g]
            dp = do[b, h] @ v[b, g].T
            out["P"][b, h], out["O"][b, h], out["dP"][b, h] = p, o, dp
            out["dS"][b, h] = p * (dp - (do[b, h] * o).sum(axis=1)[:, None])
    return out


def emulated_bwd(case, x, eps):
    """The backward evaluated in float64 with relative perturbations `eps` at
    the rounding points of a bf16 evaluation (see the module docstring)."""
    q, k, v, do = x
    B, Hq, Hkv, T, S, D = case[:6]
    G, sc = Hq // Hkv, 1.0 / np.sqrt(D)
    it = intermediates(case, x)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(B):
        for h in range(Hq):
            g = h // G
            p = it["P"][b, h]
            o_r = it["O"][b, h] * (1 + eps["O"][b, h])
            delta = (do[b, h] * o_r).sum(axis=1)
            ds = p * (it["dP"][b, h] - delta[:, None]) * (1 + eps["S"][b, h])
            dv[b, g] += (p * (1 + eps["P"][b, h])).T @ do[b, h]
            dq[b, h] = sc * (ds @ k[b, g]) * (1 + eps["dQ"][b, h])
            dk[b, g] += sc * ds.T @ q[b, h]
    return dq, dk * (1 + eps["dK"]), dv * (1 + eps["dV"])


def worst_case_eps(case, x, which, idx):
    """Roundings of at most U, each aligned in sign with its first-order
    effect on the element `idx` of gradient `which` ("dq", "dk" or "dv")."""
    q, k, v, do = x
    B, Hq, Hkv, T, S, D = case[:6]
    G, sc = Hq // Hkv, 1.0 / np.sqrt(D)
    it = intermediates(case, x)
    e = zero_eps(case)
    ref = oracle.attn_bwd_np(q, k, v, do, **_kw(case))
    if which == "dq":
        b, h, i, d = idx
        g = h // G
        e["S"][b, h, i] = U * np.sign(it["dS"][b, h, i] * k[b, g, :, d])
        # delta_i moves by sum_d' dO O eps_O: push it against sum_j P_ij K_jd
        pk = (it["P"][b, h, i] * k[b, g, :, d]).sum()
        e["O"][b, h, i] = -U * np.sign(do[b, h, i] * it["O"][b, h, i]) * np.sign(pk)
        e["dQ"][idx] = U * np.sign(ref[0][idx])
    elif which == "dk":
        b, g, j, d = idx
        for h in range(g * G, (g + 1) * G):
            e["S"][b, h, :, j] = U * np.sign(it["dS"][b, h, :, j] * q[b, h, :, d])
            # each row's delta moves against P_ij Q_id (P >= 0: against Q_id)
            e["O"][b, h] = -U * np.sign(do[b, h] * it["O"][b, h]) * \
                np.sign(q[b, h, :, d])[:, None]
        e["dK"][idx] = U * np.sign(ref[1][idx])
    else:
        b, g, j, d = idx
        for h in range(g * G, (g + 1) * G):
            e["P"][b, h, :, j] = U * np.sign(do[b, h, :, d])
        e["dV"][idx] = U * np.sign(ref[2][idx])
    return e


def _elements(shape, n, rng):
    return [tuple(int(rng.integers(0, s)) for s in shape) for _ in range(n)]


def pin_random_roundings(mag_fn, case, seed=11, draws=40):
    x = _inputs(case, seed)
    kw = _kw(case)
    A = mag_fn(*x, **kw)
    clean = emulated_bwd(case, x, zero_eps(case))
    rng = np.random.default_rng(seed + 1)
    for _ in range(draws):
        e = {n: rng.uniform(-U, U, a.shape) for n, a in zero_eps(case).items()}
        got = emulated_bwd(case, x, e)
        for name, gv, cv, a in zip(("dq", "dk", "dv"), got, clean, A):
            excess = np.abs(gv - cv) - U * a * (1 + 4 * U)
            assert excess.max() <= 1e-15, f"{name}: random rounding beyond u*A by {excess.max():.3g}"


def pin_worst_case_roundings(mag_fn, case, seed=12, per_tensor=10):
    """Aligned roundings stay within u*A and reach a good part of it."""
    x = _inputs(case, seed)
    kw = _kw(case)
    A = mag_fn(*x, **kw)
    clean = emulated_bwd(case, x, zero_eps(case))
    rng = np.random.default_rng(seed + 1)
    ratios = {"dq": [], "dk": [], "dv": []}
    for t, name in enumerate(("dq", "dk", "dv")):
        for idx in _elements(A[t].shape, per_tensor, rng):
            if A[t][idx] == 0:
                continue
            got = emulated_bwd(case, x, worst_case_eps(case, x, name, idx))
            err = abs(got[t][idx] - clean[t][idx])
            assert err <= U * A[t][idx] * (1 + 4 * U) + 1e-15, \
                f"{name}{idx}: aligned roundings move it by {err / U:.4g} u > A = {A[t][idx]:.4g}"
            ratios[name].append(err / (U * A[t][idx]))
    # The dK and dV bounds are reached term by term; dQ's delta term bounds
    # |sum_j P_ij K_jd| by sum_j P_ij |K_jd|, so its bound is reached less.
    assert np.mean(ratios["dk"]) >= 0.95 and np.mean(ratios["dv"]) >= 0.95, ratios
    assert np.mean(ratios["dq"]) >= 0.6, ratios


PINS = [pin_random_roundings, pin_worst_case_roundings]


def test_emulation_without_roundings_is_the_oracle_backward():
    for case in CASES:
        x = _inputs(case, 5)
        got = emulated_bwd(case, x, zero_eps(case))
        ref = oracle.attn_bwd_np(*x, **_kw(case))
        for gv, rv in zip(got, ref[:3]):
            assert np.allclose(gv, rv, atol=1e-12)


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) + f"-c{int(c[6])}")
@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_magnitudes_pin(pin, case):
    pin(oracle.attn_bwd_magnitudes_np, case)


# ------------------------------------------------------- planted mistakes

def _small_magnitudes(mistake=None):
    """A small, separate copy of the magnitude formula for planted mistakes."""
    def fn(q, k, v, do, causal=False, key_lens=None, q_pos=None):
        B, Hq, T, D = q.shape
        _, Hkv, S, _ = k.shape
        G, sc = Hq // Hkv, 1.0 / np.sqrt(D)
        dq, dk, dv, o, _ = oracle.attn_bwd_np(q, k, v, do, causal=causal, key_lens=key_lens,
                                              q_pos=q_pos)
        aq, ak, av = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
        for b in range(B):
            L = S if key_lens is None else int(key_lens[b])
            qp = None if q_pos is None else int(q_pos[b])
            _, vis = oracle.visibility(T, S, L, causal, qp)
            for h in range(Hq):
                g = h // G
                p = _softmax_rows(sc * q[b, h] @ k[b, g].T, vis)
                dp = do[b, h] @ v[b, g].T
                ds = np.abs(p * (dp - (do[b, h] * o[b, h]).sum(axis=1)[:, None]))
                if mistake == "p_for_ds":
                    ds = p
                rdo = np.abs(do[b, h] * o[b, h]).sum(axis=1)
                if mistake == "no_delta":
                    rdo = 0 * rdo
                aq[b, h] = sc * (ds @ np.abs(k[b, g]) + (p @ np.abs(k[b, g])) * rdo[:, None])
                ak[b, g] += sc * (ds.T @ np.abs(q[b, h]) + p.T @ (np.abs(q[b, h]) * rdo[:, None]))
                if mistake != "no_p_dv":
                    av[b, g] += p.T @ np.abs(do[b, h])
        if mistake == "no_result":
            return aq, ak, av
        res = aq + np.abs(dq), ak + np.abs(dk), av + np.abs(dv)
        if mistake == "doubled":
            res = tuple(2 * r for r in res)
        return res
    return fn


def test_clean_small_copy_passes_pins():
    for case in CASES[:2]:
        for pin in PINS:
            pin(_small_magnitudes(), case)


@pytest.mark.parametrize("mistake", ["no_delta", "no_result", "p_for_ds", "no_p_dv", "doubled"])
def test_pins_catch_planted_mistakes(mistake):
    failed = 0
    for case in CASES[:2]:
        for pin in PINS:
            try:
                pin(_small_magnitudes(mistake), case)
            except AssertionError:
                failed += 1
    assert failed >= 1, f"no pin noticed {mistake}"
