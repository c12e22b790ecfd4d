"""GPU parity of the bf16 tensor-core prefill (tcgen05 + TMA) on small cases.

Sizes span several 128x128 tiles with ragged tails in both T and S, causal
and non-causal masks, bottom-right alignment (T < S and T > S), key padding
with padded query rows, GQA, and D in {64, 128}.
"""
from __future__ import annotations

import math

import pytest
import torch

import workloads
from parity import compare, oracle_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


def _run(E, B, Hq, Hkv, T, S, D, causal, lens, seed=1, q_scale=1.0, out_rounding=False):
    x = workloads.prefill_inputs(B, Hq, Hkv, T, S, D, "bf16", seed=seed, device="cuda",
                                 lens=lens, q_scale=q_scale)
    scale = 1.0 / math.sqrt(D)
    o, lse = E.attn_fwd(x["q"], x["k"], x["v"], causal=causal, key_lens=x["key_lens"],
                        scale=scale)
    torch.cuda.synchronize()
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], causal, x["key_lens"], scale)
    st = compare(o, lse, ro, rl, torch.bfloat16, f"bf16 {(B, Hq, Hkv, T, S, D, causal, lens)}",
                 out_rounding=out_rounding)
    assert E.attn_device_error(clear=True) == 0
    return st


def test_single_tile_first(E):
    """One 128x128 tile, no mask: the smallest use of every tcgen05 piece."""
    _run(E, 1, 1, 1, 128, 128, 64, False, None)


CASES = [
    (1, 1, 1, 128, 128, 128, False, None),
    (1, 2, 2, 256, 256, 64, True, None),
    (1, 2, 2, 256, 256, 128, True, None),
    (2, 4, 2, 300, 300, 64, True, None),
    (2, 4, 1, 200, 333, 128, True, (50, 333)),
    (1, 2, 2, 333, 200, 128, True, None),
    (2, 2, 2, 129, 257, 64, False, (1, 257)),
    (1, 1, 1, 1, 1, 128, False, None),
    (2, 8, 2, 513, 513, 128, True, (200, 513)),
    (1, 2, 2, 77, 1000, 64, False, None),
    (3, 4, 4, 640, 640, 128, True, (0, 640)),
    # odd B, Hq and group size: the work walk divides by B, Hq and Hq / Hkv
    (3, 6, 2, 700, 700, 64, True, (100, 700)),
    (5, 3, 3, 300, 300, 128, True, None),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "x".join(map(str, c[:6])) +
                         f"-c{int(c[6])}-{'pad' if c[7] else 'nopad'}")
def test_prefill_bf16(E, case):
    _run(E, *case)


@pytest.mark.parametrize("q_scale", [2.0, 8.0])
def test_large_scores_rescale(E, q_scale):
    """Larger query scale makes the running maximum move often, exercising
    the lazy O rescale.  With Q x 8 the softmax is nearly one-hot and |O|
    exceeds 2, where storing O in bf16 alone can cost 1.56e-2, so that case
    allows half a bf16 ulp of the exact value on top of the tolerance."""
    _run(E, 1, 4, 4, 384, 384, 128, True, None, seed=9, q_scale=q_scale,
         out_rounding=q_scale > 4)


def test_output_buffer_and_no_lse(E):
    x = workloads.prefill_inputs(1, 2, 2, 200, 200, 64, "bf16", seed=3, device="cuda")
    o = torch.full_like(x["q"], float("nan"))
    E.attn_fwd(x["q"], x["k"], x["v"], o=o, causal=True, return_lse=False)
    torch.cuda.synchronize()
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], True, None, 1 / 8)
    compare(o, None, ro, rl, torch.bfloat16, "preallocated o")


def test_output_view_16_byte_aligned(E):
    """An output view that starts 16 bytes (not 32) into its allocation takes
    the 128-bit store path of the epilogue; results must not change."""
    x = workloads.prefill_inputs(2, 2, 2, 300, 300, 128, "bf16", seed=4, device="cuda")
    n = x["q"].numel()
    buf = torch.full((n + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
    o = buf[8:].view(x["q"].shape)
    assert o.data_ptr() % 32 == 16
    E.attn_fwd(x["q"], x["k"], x["v"], o=o, causal=True, return_lse=False)
    torch.cuda.synchronize()
    ro, rl = oracle_fwd(x["q"], x["k"], x["v"], True, None, 1 / math.sqrt(128))
    compare(o, None, ro, rl, torch.bfloat16, "16-byte aligned o")
    assert torch.isnan(buf[:8].float()).all()
