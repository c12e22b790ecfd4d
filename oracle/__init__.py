"""Float64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it,
and it shares no code with the CUDA path.

Two independent implementations of the same plain definition live here:

* ``liboracle.so`` (``attn_oracle.c``): row-by-row C, pthreads, float64.
* ``oracle_np``: vectorised NumPy float64, plus the tiled online-softmax
  recurrence used only for the "tiled == full" check.

Inputs are NumPy arrays of float64, float32 or raw bfloat16 bit patterns
(uint16, pass ``bf16=True``); each element is widened exactly to float64.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .oracle_np import (attn_bwd_magnitudes_np, attn_bwd_np, attn_decode_np, attn_fwd_fp8_np,
                        attn_fwd_kv_shard_np, attn_fwd_np, attn_tiled_online_np,
                        bf16_bits_to_f64, e4m3_bits_to_f64, lse_merge_np, visibility)

__all__ = [
    "attn_fwd", "attn_decode", "kv_append", "attn_fwd_np", "attn_decode_np", "attn_bwd_np",
    "attn_bwd_magnitudes_np", "attn_fwd_fp8_np", "e4m3_bits_to_f64", "attn_fwd_kv_shard_np",
    "lse_merge_np",
    "attn_tiled_online_np", "bf16_bits_to_f64", "visibility", "build",
    "default_threads",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "attn_oracle.c")
_lib = None

_F64, _F32, _BF16 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so (gcc, -O2, no fast-math)."""
    from .build import build_oracle
    return build_oracle(force=force)


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if (not os.path.exists(_SO)
            or os.path.getmtime(_SO) < os.path.getmtime(_SRC)):
        build()
    lib = ctypes.CDLL(_SO)
    P = ctypes.c_void_p
    I = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [P, P, P, I, I, I, I, I, I, I, I, P, P,
                                    ctypes.c_double, P, ctypes.c_int64, P, P, I]
    lib.oracle_attn_fwd.restype = I
    lib.oracle_attn_decode.argtypes = [P, P, P, I, P, I, I, I, I, I,
                                       ctypes.c_double, P, P, I]
    lib.oracle_attn_decode.restype = I
    lib.oracle_kv_append.argtypes = [P, P, P, P, P, I, I, I, I, I]
    lib.oracle_kv_append.restype = I
    _lib = lib
    return lib


def default_threads() -> int:
    """Host threads the oracle uses: the cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _prep(x: np.ndarray, bf16: bool):
    if bf16:
        a = np.ascontiguousarray(x, dtype=np.uint16)
        return a, _BF16
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), _F32
    return np.ascontiguousarray(x, dtype=np.float64), _F64


def _ptr(a) -> ctypes.c_void_p:
    return ctypes.c_void_p(a.ctypes.data) if a is not None else None


def attn_fwd(q, k, v, causal=False, key_lens=None, scale=None, bf16=False,
             rows=None, nthreads=None, q_pos=None):
    """Prefill forward by the C oracle.

    q [B,Hq,T,D], k/v [B,Hkv,S,D].  ``rows`` (optional) is an int64 array of
    flat row ids ``(b*Hq + h)*T + i``; then only those rows are computed and
    the result is packed as o [n,D], lse [n].  Otherwise o [B,Hq,T,D],
    lse [B,Hq,T].  ``q_pos`` (optional, [B]) puts query row i of sequence b
    at key position q_pos[b] + i (chunked prefill against a cache; default
    S - T, bottom-right).  Returns float64 arrays.
    """
    lib = _load()
    B, Hq, T, D = q.shape
    Bk, Hkv, S, Dk = k.shape
    if Bk != B or Dk != D or v.shape != k.shape:
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    qa, dt = _prep(q, bf16)
    ka, _ = _prep(k, bf16)
    va, _ = _prep(v, bf16)
    lens = None
    if key_lens is not None:
        lens = np.ascontiguousarray(key_lens, dtype=np.int32)
    qp = None
    if q_pos is not None:
        qp = np.ascontiguousarray(q_pos, dtype=np.int32)
        if qp.shape != (B,):
            raise ValueError("q_pos must have one entry per sequence")
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows.shape[0]
        o = np.empty((n, D))
        lse = np.empty(n)
    else:
        n = 0
        o = np.empty((B, Hq, T, D))
        lse = np.empty((B, Hq, T))
    rc = lib.oracle_attn_fwd(_ptr(qa), _ptr(ka), _ptr(va), dt, B, Hq, Hkv, T,
                             S, D, int(bool(causal)), _ptr(lens), _ptr(qp),
                             float(scale), _ptr(rows), n, _ptr(o), _ptr(lse),
                             nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd rejected its arguments (rc={rc})")
    return o, lse


def attn_decode(q, kcache, vcache, kv_lens, scale=None, bf16=False,
                nthreads=None):
    """Single-query decode by the C oracle.  q [B,Hq,D], caches
    [B,Hkv,S_max,D], kv_lens [B].  Returns (o [B,Hq,D], lse [B,Hq])."""
    lib = _load()
    B, Hq, D = q.shape
    _, Hkv, S_max, _ = kcache.shape
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    qa, dt = _prep(q, bf16)
    ka, _ = _prep(kcache, bf16)
    va, _ = _prep(vcache, bf16)
    lens = np.ascontiguousarray(kv_lens, dtype=np.int32)
    o = np.empty((B, Hq, D))
    lse = np.empty((B, Hq))
    rc = lib.oracle_attn_decode(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(lens),
                                B, Hq, Hkv, S_max, D, float(scale), _ptr(o),
                                _ptr(lse), nthreads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle_attn_decode rejected its arguments (rc={rc})")
    return o, lse


def kv_append(kcache, vcache, k_new, v_new, pos):
    """In-place append of one token per (b, kv head) at pos[b] (NumPy arrays
    of any 2- or 4-byte dtype).  Returns the number of skipped (b, g) pairs
    whose pos was outside [0, S_max)."""
    lib = _load()
    B, Hkv, S_max, D = kcache.shape
    for a in (kcache, vcache):
        if not a.flags.c_contiguous:
            raise ValueError("cache must be C-contiguous")
    kn = np.ascontiguousarray(k_new)
    vn = np.ascontiguousarray(v_new)
    p = np.ascontiguousarray(pos, dtype=np.int32)
    return lib.oracle_kv_append(_ptr(kcache), _ptr(vcache), _ptr(kn), _ptr(vn),
                                _ptr(p), B, Hkv, S_max, D,
                                kcache.dtype.itemsize)
