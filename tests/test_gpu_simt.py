"""GPU parity: exact float32 prefill, KV-cache append and split-KV decode.

Every case runs through the C ABI (via the ctypes binding) on seeded inputs
and is compared element by element with the float64 oracle.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import workloads
from parity import compare, oracle_decode, oracle_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    assert torch.cuda.is_available()
    return m


def _no_device_error(E):
    assert E.attn_device_error(clear=True) == 0


# ------------------------------------------------------------ fp32 prefill

F32_CASES = [
    # B, Hq, Hkv, T, S, D, causal, lens
    (2, 4, 2, 70, 70, 64, True, None),
    (2, 4, 2, 37, 90, 128, True, (10, 90)),
    (1, 2, 1, 90, 37, 32, True, None),
    (2, 2, 2, 33, 65, 256, False, (1, 65)),
    (1, 1, 1, 1, 1, 16, False, None),
    (3, 6, 3, 50, 50, 48, True, (0, 50)),
    (1, 3, 1, 41, 41, 7, False, None),
]


@pytest.mark.parametrize("case", F32_CASES, ids=lambda c: "x".join(map(str, c[:6])) +
                         f"-c{int(c[6])}-{'pad' if c[7] else 'nopad'}")
def test_fp32_prefill(E, case):
    B, Hq, Hkv, T, S, D, causal, lens = case
    x = workloads.prefill_inputs(B, Hq, Hkv, T, S, D, "f32", seed=100 + T, device="cuda",
                                 lens=lens)
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd(x["q"], x["k"], x["v"], causal=causal, key_lens=x["key_lens"],
                        scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], causal, x["key_lens"], scale)
    compare(o, lse, ro, rl, torch.float32, f"fp32 {case}")
    _no_device_error(E)


def test_fp32_without_lse(E):
    x = workloads.prefill_inputs(1, 2, 2, 40, 40, 64, "f32", seed=7, device="cuda")
    o, lse = E.attn_fwd(x["q"], x["k"], x["v"], causal=True, return_lse=False)
    assert lse is None
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], True, None, 1 / 8)
    compare(o, None, ro, rl, torch.float32, "fp32 no lse")


# ------------------------------------------------------------------ append

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_append_is_exact_and_bounds_checked(E, dtype):
    d = workloads.decode_inputs(3, 4, 2, 128, 5, 40, dtype, seed=3, device="cuda")
    kc, vc = d["kcache"].clone(), d["vcache"].clone()
    pos = d["cache_len"].clone()
    pos[1] = d["S_max"]          # out of range: must be skipped and reported
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.kv_cache_append(kc, vc, d["k_new"], d["v_new"], pos, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1
    want_k, want_v = d["kcache"].clone(), d["vcache"].clone()
    for b in range(3):
        p = int(pos[b])
        if 0 <= p < d["S_max"]:
            want_k[b, :, p] = d["k_new"][b]
            want_v[b, :, p] = d["v_new"][b]
    assert torch.equal(kc, want_k) and torch.equal(vc, want_v)
    assert E.attn_kernel_launches() > 0


# ------------------------------------------------------------------ decode

DEC_CASES = [
    # B, Hq, Hkv, D, lo, hi, dtype
    (3, 8, 2, 128, 1, 600, "bf16"),
    (4, 4, 4, 64, 200, 1000, "f32"),
    (2, 16, 1, 128, 255, 257, "bf16"),
    (5, 8, 4, 64, 1, 3, "bf16"),
    (2, 4, 1, 128, 511, 513, "f32"),
    (3, 32, 8, 128, 700, 2100, "bf16"),
]


@pytest.mark.parametrize("case", DEC_CASES, ids=lambda c: "-".join(map(str, c)))
def test_decode(E, case):
    B, Hq, Hkv, D, lo, hi, dtype = case
    d = workloads.decode_inputs(B, Hq, Hkv, D, lo, hi, dtype, seed=11 + B, device="cuda")
    kc, vc = d["kcache"], d["vcache"]
    E.kv_cache_append(kc, vc, d["k_new"], d["v_new"], d["cache_len"])
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_decode(d["q"], kc, vc, d["kv_len"], scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle_decode(d["q"], kc, vc, d["kv_len"], scale)
    compare(o, lse, ro, rl, torch.float32 if dtype == "f32" else torch.bfloat16,
            f"decode {case}")
    _no_device_error(E)


def test_decode_empty_sequence(E):
    d = workloads.decode_inputs(3, 4, 2, 64, 10, 20, "bf16", seed=5, device="cuda")
    kv = d["kv_len"].clone()
    kv[1] = 0
    o, lse = E.attn_decode(d["q"], d["kcache"], d["vcache"], kv)
    torch.cuda.synchronize()
    ro, rl = oracle_decode(d["q"], d["kcache"], d["vcache"], kv, 1 / 8)
    compare(o, lse, ro, rl, torch.bfloat16, "decode with an empty sequence")
    assert torch.all(o[1] == 0) and torch.all(torch.isneginf(lse[1]))


def test_incremental_decode_equals_full_forward(E):
    """Appending token t and decoding it gives row t of the causal forward
    ("Implementing attention from scratch", Testing against a reference)."""
    B, Hq, Hkv, D, n = 2, 8, 2, 64, 300
    x = workloads.prefill_inputs(B, Hq, Hkv, n, n, D, "f32", seed=21, device="cuda")
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], True, None, 1 / 8)
    kc = torch.zeros(B, Hkv, n, D, device="cuda")
    vc = torch.zeros_like(kc)
    for t in range(n):
        pos = torch.full((B,), t, dtype=torch.int32, device="cuda")
        E.kv_cache_append(kc, vc, x["k"][:, :, t].contiguous(), x["v"][:, :, t].contiguous(), pos)
        if t % 37 == 0 or t == n - 1:
            o, lse = E.attn_decode(x["q"][:, :, t].contiguous(), kc, vc, pos + 1)
            torch.cuda.synchronize()
            compare(o, lse, ro[:, :, t], rl[:, :, t], torch.float32, f"step {t}")
    assert torch.equal(kc, x["k"]) and torch.equal(vc, x["v"])
