"""The decode entry point that allocates nothing, checked against attn_decode
and against the float64 oracle.

attn_decode_noalloc is for callers that cannot allocate device memory: a
host framework that owns every byte of it through its own allocator, or a
real-time loop that cannot afford cudaMalloc's device synchronisation.  It
uses a fixed scratch array that the library defines in device memory instead
of a caller-provided workspace.  It runs the same kernels on the same inputs
as attn_decode, and those kernels are deterministic (the work split depends
only on the lengths and the SM count), so its outputs must be bit-identical
to attn_decode's.  Two calls in a row with different shapes and dtypes make
the second call find the first one's leftovers in the shared array; each
call is also compared with the float64 oracle within the parity tolerances.
"""
from __future__ import annotations

import math

import pytest
import torch

import workloads
from parity import compare, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


CALLS = [
    # B, Hq, Hkv, D, lo, hi, dtype, seed
    (4, 16, 4, 128, 300, 1500, "bf16", 31),
    (3, 8, 8, 64, 1, 2000, "f32", 32),
]


def test_noalloc_matches_decode_on_two_calls_in_a_row(E):
    for B, Hq, Hkv, D, lo, hi, dtype, seed in CALLS:
        d = workloads.decode_inputs(B, Hq, Hkv, D, lo, hi, dtype, seed=seed, device="cuda")
        scale = 1.0 / math.sqrt(D)
        ref_o, ref_l = E.attn_decode(d["q"], d["kcache"], d["vcache"], d["kv_len"], scale=scale)
        o = torch.full_like(d["q"], float("nan"))
        lse = torch.full((B, Hq), float("nan"), device="cuda")
        E.attn_decode_noalloc(d["q"], d["kcache"], d["vcache"], d["kv_len"], o, lse,
                              scale=scale)
        torch.cuda.synchronize()
        assert E.attn_device_error(clear=True) == 0
        # same kernels, same inputs: the same bits
        assert torch.equal(o.view(torch.int16 if o.dtype != torch.float32 else torch.int32),
                           ref_o.view(torch.int16 if o.dtype != torch.float32 else torch.int32))
        assert torch.equal(lse.view(torch.int32), ref_l.view(torch.int32))
        # and the float64 oracle on the same input values
        ro, rl = oracle_decode(d["q"], d["kcache"], d["vcache"], d["kv_len"], scale)
        compare(o, lse, ro, rl, d["q"].dtype, f"noalloc decode {dtype} D{D}")


def test_noalloc_rejects_requests_beyond_its_scratch(E):
    # 64 x 32 heads x 34 slots x (128 + 2) floats = 36 MB > 16 MiB
    need = E.attn_decode_workspace_size(64, 32, 8193, 128)
    assert need > E.NOALLOC_SCRATCH_BYTES
    q = torch.zeros(64, 32, 128, device="cuda", dtype=torch.bfloat16)
    kc = torch.zeros(64, 8, 8193, 128, device="cuda", dtype=torch.bfloat16)
    kv = torch.full((64,), 10, device="cuda", dtype=torch.int32)
    o = torch.empty_like(q)
    before = E.attn_kernel_launches()
    with pytest.raises(E.AttnError) as info:
        E.attn_decode_noalloc(q, kc, kc, kv, o)
    assert info.value.status == E.ATTN_ERR_WORKSPACE
    assert E.attn_kernel_launches() == before
