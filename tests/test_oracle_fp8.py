"""Pins of the FP8 (E4M3) part of the oracle, on the CPU.

The decoder is checked against values fixed by the format's definition
(closed forms), against PyTorch's own float8_e4m3fn widening for all 256
codes (a library routine, independent of ours), and for order.  The FP8
attention oracle is checked through invariants of the definition that a
wrong scale, operand or mask would break.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x40, 2.0), (0x3C, 1.5), (0x30, 0.5), (0x7E, 448.0),
    (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x08, 2.0 ** -6), (0x77, 240.0),
    (0xB8, -1.0), (0xFE, -448.0), (0x81, -(2.0 ** -9)),
])
def test_e4m3_closed_forms(code, value):
    assert oracle.e4m3_bits_to_f64(np.array([code], dtype=np.uint8))[0] == value


def test_e4m3_nan_and_negative_zero():
    v = oracle.e4m3_bits_to_f64(np.array([0x7F, 0xFF, 0x80], dtype=np.uint8))
    assert np.isnan(v[0]) and np.isnan(v[1])
    assert v[2] == 0.0 and math.copysign(1.0, v[2]) < 0


def test_e4m3_matches_torch_for_every_code():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_bits_to_f64(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all(), codes[~same]


def test_e4m3_positive_codes_increase():
    v = oracle.e4m3_bits_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)


def _rand_fp8(rng, shape):
    x = torch.from_numpy(rng.standard_normal(shape)).float()
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_fp8_attention_descale_invariants():
    rng = np.random.default_rng(5)
    q8, k8, v8 = (_rand_fp8(rng, (1, 2, 37, 16)) for _ in range(3))
    o1, l1 = oracle.attn_fwd_fp8_np(q8, k8, v8, causal=True, scale=0.25)
    # V's scale scales O and leaves LSE
    o2, l2 = oracle.attn_fwd_fp8_np(q8, k8, v8, v_descale=2.0, causal=True, scale=0.25)
    np.testing.assert_array_equal(o2, 2.0 * o1)
    np.testing.assert_array_equal(l2, l1)
    # a scale on Q traded against the softmax scale changes nothing
    o3, l3 = oracle.attn_fwd_fp8_np(q8, k8, v8, q_descale=4.0, causal=True, scale=0.0625)
    np.testing.assert_allclose(o3, o1, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l3, l1, rtol=0, atol=1e-12)


def test_fp8_attention_identical_value_rows():
    rng = np.random.default_rng(6)
    q8, k8 = (_rand_fp8(rng, (1, 1, 20, 16)) for _ in range(2))
    row = _rand_fp8(rng, (16,))
    v8 = np.broadcast_to(row, (1, 1, 20, 16)).copy()
    o, _ = oracle.attn_fwd_fp8_np(q8, k8, v8, v_descale=0.5, scale=0.3)
    expect = oracle.e4m3_bits_to_f64(row) * 0.5
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(expect, (20, 16)), rtol=0, atol=1e-12)


def test_fp8_attention_is_bf16_definition_on_dequantised_inputs():
    """Every E4M3 value times a power of two is exact in bfloat16 (8 bits of
    precision >= 4), so the FP8 oracle must equal the bf16 oracle fed with
    the same values as bf16 bit patterns."""
    rng = np.random.default_rng(7)
    q8, k8, v8 = (_rand_fp8(rng, (2, 2, 33, 16)) for _ in range(3))
    o8, l8 = oracle.attn_fwd_fp8_np(q8, k8, v8, q_descale=0.5, k_descale=2.0, v_descale=0.25,
                                    causal=True, key_lens=np.array([33, 20]), scale=0.2)
    bits = [torch.from_numpy(oracle.e4m3_bits_to_f64(x) * s).to(torch.bfloat16).view(torch.uint16).numpy()
            for x, s in ((q8, 0.5), (k8, 2.0), (v8, 0.25))]
    ob, lb = oracle.attn_fwd(*bits, causal=True, key_lens=np.array([33, 20]), scale=0.2, bf16=True)
    valid = np.isfinite(lb)
    np.testing.assert_allclose(o8[valid], ob[valid], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l8[valid], lb[valid], rtol=0, atol=1e-12)
