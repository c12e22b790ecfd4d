"""The C-ABI library loads and exports what include/attn.h declares (CPU).

No kernel is launched here: every call below is rejected by host-side
validation before any CUDA runtime call, or is a pure host function.
"""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


@pytest.fixture(scope="module")
def lib():
    from exact_tiled_attention_49_b300 import build
    build.build()
    import exact_tiled_attention_49_b300 as m
    return m.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["attn_fwd", "attn_decode", "attn_decode_workspace_size", "kv_cache_append",
              "attn_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_covers_header():
    import exact_tiled_attention_49_b300 as m
    assert sorted(m.SIGNATURES) == declared_functions()


def test_only_declared_symbols_exported():
    from exact_tiled_attention_49_b300 import LIB_PATH
    out = subprocess.run(["nm", "-D", "--defined-only", LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines()
                if line.split() and line.split()[-2] in ("T", "W")}
    ours = {s for s in exported if s.startswith(("attn_", "kv_cache"))}
    assert ours == set(declared_functions())


def test_status_strings(lib):
    for code in range(5):
        s = lib.attn_status_string(code).decode()
        assert s.startswith("ATTN_")
    assert "unknown" in lib.attn_status_string(99).decode()


def test_workspace_size_formula(lib):
    # partial O (D floats) + running max + denominator per (b, h) and slot,
    # ceil(S_max / 256) + 1 slots; then B + 2 int64 of the split plan
    assert lib.attn_decode_workspace_size(64, 32, 8193, 128) == 64 * 32 * 34 * 130 * 4 + 66 * 8
    assert lib.attn_decode_workspace_size(1, 1, 256, 64) == 1 * 1 * 2 * 66 * 4 + 3 * 8
    assert lib.attn_decode_workspace_size(0, 1, 1, 64) == 0


FAKE = ctypes.c_void_p(0x10000)  # 16-byte aligned, never dereferenced
MIS = ctypes.c_void_p(0x10002)   # misaligned


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=None, B=1, Hq=1, Hkv=1, T=8, S=8, D=64,
         dt=1, causal=0, lens=None, scale=0.125):
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, T, S, D, dt, causal, lens, scale, None)


def test_fwd_rejects_bad_arguments(lib):
    assert _fwd(lib, q=None) == 1
    assert _fwd(lib, B=0) == 1
    assert _fwd(lib, T=-1) == 1
    assert _fwd(lib, Hq=3, Hkv=2) == 1
    assert _fwd(lib, scale=0.0) == 1
    assert _fwd(lib, scale=float("nan")) == 1
    assert _fwd(lib, D=96) == 2            # bf16 supports D in {64, 128}
    assert _fwd(lib, D=300, dt=0) == 2     # fp32 supports D <= 256
    assert _fwd(lib, q=MIS) == 1           # TMA needs 16-byte alignment
    assert _fwd(lib, dt=7) == 1


def test_decode_rejects_bad_arguments(lib):
    ws = lib.attn_decode_workspace_size(2, 4, 100, 64)

    def dec(kv_lens=FAKE, D=64, Hq=4, Hkv=2, ws_ptr=FAKE, ws_bytes=ws, dt=1):
        return lib.attn_decode(FAKE, FAKE, FAKE, kv_lens, FAKE, None, 2, Hq, Hkv, 100, D, dt,
                               0.125, ws_ptr, ws_bytes, None)
    assert dec(kv_lens=None) == 1
    assert dec(Hq=6, Hkv=4) == 1
    assert dec(D=96) == 2
    assert dec(Hq=64, Hkv=2) == 2          # group of 32 query heads per KV head
    assert dec(ws_ptr=None) == 3
    assert dec(ws_bytes=ws - 4) == 3


def test_decode_noalloc_checks_arguments_before_its_scratch(lib):
    """attn_decode_noalloc reports an invalid or unsupported request the way
    attn_decode does, even when its workspace would exceed the fixed
    scratch array (which alone would give ATTN_ERR_WORKSPACE)."""
    big = (64, 32, 8, 100000)            # B, Hq, Hkv, S_max: far beyond the scratch

    def na(q=FAKE, D=128, Hq=32, Hkv=8, dt=1, scale=0.125):
        B, _, _, S_max = big
        return lib.attn_decode_noalloc(q, FAKE, FAKE, FAKE, FAKE, None, B, Hq, Hkv, S_max, D,
                                       dt, scale, None)
    from exact_tiled_attention_49_b300 import NOALLOC_SCRATCH_BYTES
    assert lib.attn_decode_workspace_size(64, 32, 100000, 96) > NOALLOC_SCRATCH_BYTES
    assert na(D=96) == 2                   # unsupported head size, not "too large"
    assert na(q=None) == 1                 # invalid argument, not "too large"
    assert na(Hq=6, Hkv=4) == 1
    assert na(dt=7) == 1
    assert na(scale=0.0) == 1
    assert na(q=MIS) == 1
    assert na() == 3                       # a valid request that does not fit


def test_append_rejects_bad_arguments(lib):
    def app(D=64, dt=1, pos=FAKE, k=FAKE):
        return lib.kv_cache_append(k, FAKE, FAKE, FAKE, pos, 2, 2, 10, D, dt, None, None)
    assert app(pos=None) == 1
    assert app(D=4) == 1                   # 8-byte rows cannot be copied as 16-byte vectors
    assert app(k=MIS) == 1
    assert app(dt=5) == 1


def test_launch_counter_is_host_side(lib):
    assert isinstance(lib.attn_kernel_launches(), int)


def test_fwd_fp8_rejects_bad_arguments(lib):
    def f8(q=FAKE, D=128, Hq=2, Hkv=1, qd=0.5, kd=0.5, vd=0.5, scale=0.125):
        return lib.attn_fwd_fp8(q, FAKE, FAKE, FAKE, None, 1, Hq, Hkv, 8, 8, D, 1, None, scale,
                                qd, kd, vd, None)
    assert f8(q=None) == 1
    assert f8(Hq=3, Hkv=2) == 1
    assert f8(qd=0.0) == 1                 # descales must be finite and > 0
    assert f8(vd=float("nan")) == 1
    assert f8(kd=-1.0) == 1
    assert f8(scale=float("inf")) == 1
    assert f8(D=64) == 2                   # E4M3 rows must be one 128-byte swizzle row
    assert f8(q=MIS) == 1


def test_fwd_chunked_rejects_bad_arguments(lib):
    def ch(q_pos=FAKE, kv_lens=FAKE, D=64, dt=1):
        return lib.attn_fwd_chunked(FAKE, FAKE, FAKE, FAKE, None, q_pos, kv_lens, 1, 1, 1, 8, 16,
                                    D, dt, 1, 0.125, None)
    assert ch(q_pos=None) == 1             # q_pos and kv_lens are required
    assert ch(kv_lens=None) == 1
    assert ch(D=96) == 2
    assert ch(dt=7) == 1


def test_bwd_rejects_bad_arguments(lib):
    need = lib.attn_bwd_workspace_size(1, 2, 8)
    assert need >= 2 * 8 * 4               # one fp32 delta per query row

    def bw(dq=FAKE, D=64, dt=1, ws=FAKE, ws_bytes=need, Hq=2, Hkv=1):
        return lib.attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, dq, FAKE, FAKE, 1, Hq, Hkv, 8, 8, D,
                            dt, 1, None, None, 0.125, ws, ws_bytes, None)
    assert bw(dq=None) == 1
    assert bw(Hq=3, Hkv=2) == 1
    assert bw(dt=0, D=300) == 2            # fp32: D <= 256
    assert bw(dt=0, dq=MIS) == 1           # fp32: 4-byte alignment
    assert bw(dt=0, ws=None) == 3
    assert bw(D=96) == 2                   # bf16 / fp16: D in {64, 128}
    assert bw(ws=None) == 3
    assert bw(ws_bytes=need - 4) == 3


def test_kv_shard_and_merge_reject_bad_arguments(lib):
    def sh(q_pos=FAKE, key_lens=FAKE, k_off=0, D=64, dt=1, Hq=2, Hkv=1):
        return lib.attn_fwd_kv_shard(FAKE, FAKE, FAKE, FAKE, None, q_pos, key_lens, k_off, 1, Hq,
                                     Hkv, 8, 16, D, dt, 1, 0.125, None)
    assert sh(q_pos=None) == 1             # global positions are required
    assert sh(key_lens=None) == 1
    assert sh(k_off=-1) == 1
    assert sh(k_off=1 << 30) == 2          # positions are limited to 2^30
    assert sh(Hq=3, Hkv=2) == 1
    assert sh(D=96) == 2
    assert sh(dt=7) == 1

    def mg(o_parts=FAKE, n=2, D=64, dt=1, o=FAKE):
        return lib.attn_lse_merge(o_parts, FAKE, n, o, None, 1, 2, 8, D, dt, None)
    assert mg(o_parts=None) == 1
    assert mg(n=0) == 1
    assert mg(dt=9) == 1
    assert mg(D=4) == 2                    # 8-byte rows cannot be merged as 16-byte vectors
    assert mg(o=MIS) == 1


def test_fwd_host_workspace_and_rejections(lib):
    # q, k, v, o, lse and key_lens at 256-byte aligned offsets
    a = lambda x: (x + 255) // 256 * 256
    B, Hq, Hkv, T, S, D = 3, 8, 2, 100, 130, 64
    want = 2 * a(B * Hq * T * D * 2) + 2 * a(B * Hkv * S * D * 2) + a(B * Hq * T * 4) + a(B * 4)
    assert lib.attn_fwd_host_workspace_size(B, Hq, Hkv, T, S, D, 1) == want
    assert lib.attn_fwd_host_workspace_size(B, Hq, Hkv, T, S, D, 0) == \
        2 * a(B * Hq * T * D * 4) + 2 * a(B * Hkv * S * D * 4) + a(B * Hq * T * 4) + a(B * 4)
    assert lib.attn_fwd_host_workspace_size(0, 1, 1, 8, 8, 64, 1) == 0
    assert lib.attn_fwd_host_workspace_size(1, 1, 1, 8, 8, 96, 1) == 0   # unsupported D
    need = lib.attn_fwd_host_workspace_size(1, 2, 1, 8, 8, 64, 1)

    def fh(q=FAKE, ws=FAKE, ws_bytes=need, D=64, dt=1, Hq=2, Hkv=1, scale=0.125):
        return lib.attn_fwd_host(q, FAKE, FAKE, FAKE, None, 1, Hq, Hkv, 8, 8, D, dt, 1, None,
                                 scale, ws, ws_bytes, None, None, None)
    assert fh(q=None) == 1
    assert fh(Hq=3, Hkv=2) == 1
    assert fh(scale=-1.0) == 1
    assert fh(dt=5) == 1
    assert fh(D=96) == 2
    assert fh(ws=None) == 3
    assert fh(ws_bytes=need - 1) == 3
    assert fh(ws=MIS) == 3


def test_decode_append_rejects_bad_arguments(lib):
    need = lib.attn_decode_workspace_size(1, 2, 64, 64)

    def da(kn=FAKE, vn=FAKE, D=64, dt=1, ws=FAKE, ws_bytes=need, q=FAKE):
        return lib.attn_decode_append(q, FAKE, FAKE, kn, vn, FAKE, FAKE, None, 1, 2, 1, 64, D,
                                      dt, 0.125, ws, ws_bytes, None)
    assert da(q=None) == 1
    assert da(kn=None) == 1
    assert da(vn=MIS) == 1
    assert da(D=96) == 2
    assert da(dt=9) == 1
    assert da(ws=None) == 3
    assert da(ws_bytes=need - 1) == 3
