"""Failure detection on the GPU without a fault: a bounded pipeline wait
that can never complete must give up, report through the device error word,
and leave the context usable (no trap, no hang)."""
from __future__ import annotations

import math
import time

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def E():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    m.load()
    return m


def test_wait_that_never_completes_gives_up_and_reports(E):
    assert E.attn_device_error(clear=True) == 0
    t0 = time.perf_counter()
    E.attn_selftest_wait_timeout()
    code = E.attn_device_error(clear=True)     # synchronises the device
    elapsed = time.perf_counter() - t0
    assert code == E.ATTN_SELFTEST_ERROR
    assert 0.5 < elapsed < 30.0                # it waited for its limit, then returned
    assert E.attn_device_error(clear=True) == 0  # cleared

    # the context still works: a small prefill runs and reports no error
    q = torch.randn(1, 1, 128, 64, device="cuda").to(torch.bfloat16)
    o, lse = E.attn_fwd(q, q, q, causal=True, scale=1.0 / math.sqrt(64))
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert E.attn_device_error(clear=True) == 0
