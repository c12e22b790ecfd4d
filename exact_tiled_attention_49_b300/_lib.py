"""ctypes binding of libattn.so (argument marshalling only).

Every function here validates Python-side types, turns torch tensors into
device pointers and sizes, and calls the C entry point of the same name on
the current CUDA stream.  All arithmetic runs in the library's CUDA kernels;
there is no CPU or PyTorch fallback, and a missing library is an error.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE, ATTN_ERR_CUDA = range(5)
ATTN_F32, ATTN_BF16, ATTN_F16 = 0, 1, 2

# Every entry point declared in include/attn.h, with its ctypes signature.
_P, _I, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
SIGNATURES = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _F, _P]),
    "attn_fwd_chunked": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F,
                              _P]),
    "attn_fwd_fp8": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _F, _F, _F, _F,
                          _P]),
    "attn_fwd_host_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I, _I, _I]),
    "attn_fwd_host": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _F, _P,
                           ctypes.c_size_t, _P, _P, _P]),
    "attn_fwd_kv_shard": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                               _F, _P]),
    "attn_lse_merge": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P]),
    "attn_bwd_workspace_size": (ctypes.c_size_t, [_I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P,
                      _F, _P, ctypes.c_size_t, _P]),
    "attn_decode_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "attn_decode": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P,
                         ctypes.c_size_t, _P]),
    "attn_decode_append": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P,
                                ctypes.c_size_t, _P]),
    "attn_decode_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P]),
    "kv_cache_append": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_kernel_launches": (ctypes.c_ulonglong, []),
    "attn_device_error": (_I, [ctypes.POINTER(ctypes.c_int), _I]),
    "attn_selftest_wait_timeout": (_I, [_P]),
}


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def load(path: str = LIB_PATH):
    """Load libattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with `python -m exact_tiled_attention_49_b300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def attn_status_string(status: int) -> str:
    return status_string(status)


def _check(rc: int, what: str):
    if rc != ATTN_OK:
        raise AttnError(rc, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float16:
        return ATTN_F16
    if t.dtype == torch.float32:
        return ATTN_F32
    raise TypeError(f"unsupported dtype {t.dtype}; expected bfloat16, float16 or float32")


def _dev(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def attn_fwd(q, k, v, o=None, lse=None, causal=False, key_lens=None, scale=None,
             return_lse=True, stream=None):
    """Prefill forward.  q [B,Hq,T,D], k/v [B,Hkv,S,D] (bf16 or fp32, CUDA).

    Returns (o, lse): o like q, lse float32 [B,Hq,T] (None if return_lse is
    False and no lse buffer was given).  key_lens: int32 CUDA [B] or None.
    """
    lib = load()
    B, Hq, T, D = q.shape
    Bk, Hkv, S, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q/k/v shape mismatch")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, T), device=q.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ptrs = [_dev(q, "q", ndim=4), _dev(k, "k", ndim=4), _dev(v, "v", ndim=4),
            _dev(o, "o", dtype=q.dtype, ndim=4)]
    if tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must have q's shape")
    lp = None
    if lse is not None:
        lp = _dev(lse, "lse", dtype=torch.float32)
        if lse.numel() != B * Hq * T:
            raise ValueError("lse must hold B*Hq*T floats")
    kl = None
    if key_lens is not None:
        kl = _dev(key_lens, "key_lens", dtype=torch.int32, ndim=1)
        if key_lens.numel() != B:
            raise ValueError("key_lens must have B entries")
    rc = lib.attn_fwd(*ptrs, lp, B, Hq, Hkv, T, S, D, dt, int(bool(causal)), kl,
                      float(scale), _stream(stream))
    _check(rc, "attn_fwd")
    return o, lse


def _host(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions")
    return ctypes.c_void_p(t.data_ptr())


def attn_fwd_host_workspace_size(B, Hq, Hkv, T, S, D, dtype) -> int:
    code = dtype if isinstance(dtype, int) else _dtype_code(torch.empty(0, dtype=dtype))
    return int(load().attn_fwd_host_workspace_size(B, Hq, Hkv, T, S, D, code))


def attn_fwd_host(q, k, v, o=None, lse=None, causal=False, key_lens=None, scale=None,
                  return_lse=True, workspace=None, stream=None, copy_in=None, copy_out=None):
    """attn_fwd on host tensors (pinned for overlap): q [B,Hq,T,D], k/v
    [B,Hkv,S,D] and key_lens (int32 [B] or None) on the CPU; o and lse are
    written on the CPU (pinned ones are allocated when not given).  The
    library copies the inputs in, computes and copies the results out in
    pipelined stages on `stream` (compute), `copy_in` and `copy_out`
    (torch.cuda.Stream objects; None = no overlap for that role).  Returns
    (o, lse); they are complete once `stream` is."""
    lib = load()
    B, Hq, T, D = q.shape
    Bk, Hkv, S, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q/k/v shape mismatch")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, pin_memory=True)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must have q's shape")
    ptrs = [_host(q, "q", ndim=4), _host(k, "k", ndim=4), _host(v, "v", ndim=4),
            _host(o, "o", dtype=q.dtype, ndim=4)]
    lp = None
    if lse is not None:
        lp = _host(lse, "lse", dtype=torch.float32)
        if lse.numel() != B * Hq * T:
            raise ValueError("lse must hold B*Hq*T floats")
    kl = None
    if key_lens is not None:
        kl = _host(key_lens, "key_lens", dtype=torch.int32, ndim=1)
        if key_lens.numel() != B:
            raise ValueError("key_lens must have B entries")
    need = int(lib.attn_fwd_host_workspace_size(B, Hq, Hkv, T, S, D, dt))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
    wp = _dev(workspace, "workspace", dtype=torch.uint8)
    side = [None if s is None else ctypes.c_void_p(s.cuda_stream) for s in (copy_in, copy_out)]
    rc = lib.attn_fwd_host(*ptrs, lp, B, Hq, Hkv, T, S, D, dt, int(bool(causal)), kl,
                           float(scale), wp, workspace.numel(), _stream(stream), *side)
    _check(rc, "attn_fwd_host")
    return o, lse


def attn_fwd_fp8(q, k, v, o=None, lse=None, causal=False, key_lens=None, scale=None,
                 q_descale=1.0, k_descale=1.0, v_descale=1.0, return_lse=True, stream=None):
    """Prefill forward on FP8 E4M3 inputs: attention of q_descale*q,
    k_descale*k, v_descale*v.  q [B,Hq,T,128], k/v [B,Hkv,S,128] as
    torch.float8_e4m3fn (or their uint8 bytes), CUDA.  Returns (o, lse) with
    o bfloat16 [B,Hq,T,128] and lse float32 [B,Hq,T]."""
    lib = load()
    B, Hq, T, D = q.shape
    Bk, Hkv, S, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q/k/v shape mismatch")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
            raise TypeError(f"{name} must be float8_e4m3fn (or its uint8 bytes)")
    if o is None:
        o = torch.empty(q.shape, device=q.device, dtype=torch.bfloat16)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, T), device=q.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ptrs = [_dev(q, "q", ndim=4), _dev(k, "k", ndim=4), _dev(v, "v", ndim=4),
            _dev(o, "o", dtype=torch.bfloat16, ndim=4)]
    if tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must have q's shape")
    lp = None
    if lse is not None:
        lp = _dev(lse, "lse", dtype=torch.float32)
        if lse.numel() != B * Hq * T:
            raise ValueError("lse must hold B*Hq*T floats")
    kl = None
    if key_lens is not None:
        kl = _dev(key_lens, "key_lens", dtype=torch.int32, ndim=1)
        if key_lens.numel() != B:
            raise ValueError("key_lens must have B entries")
    rc = lib.attn_fwd_fp8(*ptrs, lp, B, Hq, Hkv, T, S, D, int(bool(causal)), kl, float(scale),
                          float(q_descale), float(k_descale), float(v_descale), _stream(stream))
    _check(rc, "attn_fwd_fp8")
    return o, lse


def attn_fwd_chunked(q, kcache, vcache, q_pos, kv_lens, o=None, lse=None, causal=True,
                     scale=None, return_lse=True, stream=None):
    """Chunked prefill against a KV cache.  q [B,Hq,T,D], caches
    [B,Hkv,S_max,D] (holding the chunk's own K/V rows), q_pos and kv_lens
    int32 CUDA [B]: query row i of sequence b sits at key position
    q_pos[b] + i and sees keys below kv_lens[b] (causally, up to itself).

    Returns (o, lse) like attn_fwd.
    """
    lib = load()
    B, Hq, T, D = q.shape
    Bk, Hkv, S_max, Dk = kcache.shape
    if Bk != B or Dk != D or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("q/cache shape mismatch")
    if kcache.dtype != q.dtype or vcache.dtype != q.dtype:
        raise TypeError("q and the caches must share one dtype")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, T), device=q.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    ptrs = [_dev(q, "q", ndim=4), _dev(kcache, "kcache", ndim=4),
            _dev(vcache, "vcache", ndim=4), _dev(o, "o", dtype=q.dtype, ndim=4)]
    if tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must have q's shape")
    lp = None
    if lse is not None:
        lp = _dev(lse, "lse", dtype=torch.float32)
        if lse.numel() != B * Hq * T:
            raise ValueError("lse must hold B*Hq*T floats")
    qp = _dev(q_pos, "q_pos", dtype=torch.int32, ndim=1)
    kl = _dev(kv_lens, "kv_lens", dtype=torch.int32, ndim=1)
    if q_pos.numel() != B or kv_lens.numel() != B:
        raise ValueError("q_pos and kv_lens must have B entries")
    rc = lib.attn_fwd_chunked(*ptrs, lp, qp, kl, B, Hq, Hkv, T, S_max, D, dt,
                              int(bool(causal)), float(scale), _stream(stream))
    _check(rc, "attn_fwd_chunked")
    return o, lse


def attn_fwd_kv_shard(q, k, v, q_pos, key_lens, k_off, o=None, lse=None, causal=True,
                      scale=None, stream=None):
    """Prefill over one shard of the keys.  q [B,Hq,T,D]; k/v [B,Hkv,S,D]
    hold the keys at global positions k_off .. k_off + S - 1; q_pos and
    key_lens (int32 CUDA [B]) are global: query row i of sequence b sits at
    q_pos[b] + i, keys below key_lens[b] are valid.  Returns (o, lse) of this
    shard alone, to be combined with attn_lse_merge."""
    lib = load()
    B, Hq, T, D = q.shape
    Bk, Hkv, S, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q/k/v shape mismatch")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share one dtype")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, T), device=q.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if tuple(o.shape) != tuple(q.shape) or lse.numel() != B * Hq * T:
        raise ValueError("o must have q's shape and lse B*Hq*T floats")
    if q_pos.numel() != B or key_lens.numel() != B:
        raise ValueError("q_pos and key_lens must have B entries")
    rc = lib.attn_fwd_kv_shard(_dev(q, "q", ndim=4), _dev(k, "k", ndim=4), _dev(v, "v", ndim=4),
                               _dev(o, "o", dtype=q.dtype, ndim=4),
                               _dev(lse, "lse", dtype=torch.float32),
                               _dev(q_pos, "q_pos", dtype=torch.int32, ndim=1),
                               _dev(key_lens, "key_lens", dtype=torch.int32, ndim=1),
                               int(k_off), B, Hq, Hkv, T, S, D, dt, int(bool(causal)),
                               float(scale), _stream(stream))
    _check(rc, "attn_fwd_kv_shard")
    return o, lse


def attn_lse_merge(o_parts, lse_parts, o=None, lse=None, stream=None):
    """Merge partials over disjoint key sets: o_parts [N,B,Hq,T,D] (bf16, fp16
    or fp32), lse_parts float32 [N,B,Hq,T] -> (o [B,Hq,T,D], lse [B,Hq,T])."""
    lib = load()
    N, B, Hq, T, D = o_parts.shape
    if tuple(lse_parts.shape) != (N, B, Hq, T):
        raise ValueError("lse_parts must be [N,B,Hq,T]")
    if o is None:
        o = torch.empty(o_parts.shape[1:], device=o_parts.device, dtype=o_parts.dtype)
    if lse is None:
        lse = torch.empty((B, Hq, T), device=o_parts.device, dtype=torch.float32)
    if tuple(o.shape) != tuple(o_parts.shape[1:]) or lse.numel() != B * Hq * T:
        raise ValueError("o must be [B,Hq,T,D] and lse B*Hq*T floats")
    rc = lib.attn_lse_merge(_dev(o_parts, "o_parts", ndim=5),
                            _dev(lse_parts, "lse_parts", dtype=torch.float32, ndim=4), N,
                            _dev(o, "o", dtype=o_parts.dtype, ndim=4),
                            _dev(lse, "lse", dtype=torch.float32), B, Hq, T, D,
                            _dtype_code(o_parts), _stream(stream))
    _check(rc, "attn_lse_merge")
    return o, lse


def attn_bwd_workspace_size(B: int, Hq: int, T: int) -> int:
    return int(load().attn_bwd_workspace_size(B, Hq, T))


def attn_bwd(q, k, v, o, dout, lse, causal=False, key_lens=None, q_pos=None, scale=None,
             dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward pass: (dq, dk, dv) for attn_fwd's (o, lse) and the gradient
    dout of its output.  q/o/dout [B,Hq,T,D], k/v [B,Hkv,S,D] (bf16, fp16 or
    fp32, CUDA);
    key_lens / q_pos as for attn_fwd / attn_fwd_chunked."""
    lib = load()
    B, Hq, T, D = q.shape
    Bk, Hkv, S, Dk = k.shape
    if Bk != B or Dk != D or tuple(v.shape) != tuple(k.shape):
        raise ValueError("q/k/v shape mismatch")
    for t, name in ((o, "o"), (dout, "dout")):
        if tuple(t.shape) != tuple(q.shape):
            raise ValueError(f"{name} must have q's shape")
    dt = _dtype_code(q)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    need = attn_bwd_workspace_size(B, Hq, T)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    ptrs = [_dev(q, "q", ndim=4), _dev(k, "k", ndim=4), _dev(v, "v", ndim=4),
            _dev(o, "o", dtype=q.dtype, ndim=4), _dev(dout, "dout", dtype=q.dtype, ndim=4),
            _dev(lse, "lse", dtype=torch.float32), _dev(dq, "dq", dtype=q.dtype, ndim=4),
            _dev(dk, "dk", dtype=q.dtype, ndim=4), _dev(dv, "dv", dtype=q.dtype, ndim=4)]
    if lse.numel() != B * Hq * T:
        raise ValueError("lse must hold B*Hq*T floats")
    kl = None
    if key_lens is not None:
        kl = _dev(key_lens, "key_lens", dtype=torch.int32, ndim=1)
    qp = None
    if q_pos is not None:
        qp = _dev(q_pos, "q_pos", dtype=torch.int32, ndim=1)
    rc = lib.attn_bwd(*ptrs, B, Hq, Hkv, T, S, D, dt, int(bool(causal)), kl, qp, float(scale),
                      _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                      _stream(stream))
    _check(rc, "attn_bwd")
    return dq, dk, dv


def attn_decode_workspace_size(B: int, Hq: int, S_max: int, D: int) -> int:
    return int(load().attn_decode_workspace_size(B, Hq, S_max, D))


def attn_decode(q, kcache, vcache, kv_lens, o=None, lse=None, workspace=None,
                scale=None, return_lse=True, stream=None):
    """Decode step.  q [B,Hq,D], caches [B,Hkv,S_max,D], kv_lens int32 [B].

    ``workspace`` (uint8 CUDA tensor) is allocated if not given.
    Returns (o [B,Hq,D], lse [B,Hq] or None).
    """
    lib = load()
    B, Hq, D = q.shape
    Bk, Hkv, S_max, Dk = kcache.shape
    if Bk != B or Dk != D or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("q/cache shape mismatch")
    if kcache.dtype != q.dtype or vcache.dtype != q.dtype:
        raise TypeError("q and the caches must share one dtype")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32)
    need = attn_decode_workspace_size(B, Hq, S_max, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lp = _dev(lse, "lse", dtype=torch.float32) if lse is not None else None
    rc = lib.attn_decode(_dev(q, "q", ndim=3), _dev(kcache, "kcache", ndim=4),
                         _dev(vcache, "vcache", ndim=4),
                         _dev(kv_lens, "kv_lens", dtype=torch.int32, ndim=1),
                         _dev(o, "o", dtype=q.dtype, ndim=3), lp, B, Hq, Hkv, S_max, D, dt,
                         float(scale), _dev(workspace, "workspace"),
                         workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_decode")
    return o, lse


def attn_decode_append(q, kcache, vcache, k_new, v_new, kv_lens, o=None, lse=None,
                       workspace=None, scale=None, return_lse=True, stream=None):
    """Append the new token's K/V rows (k_new, v_new [B,Hkv,D]) at row
    kv_lens[b] - 1 of the caches and decode over kv_lens[b] rows, in one
    call.  kv_lens counts the new token.  Same results as
    kv_cache_append(pos=kv_lens - 1) followed by attn_decode.
    Returns (o [B,Hq,D], lse [B,Hq] or None)."""
    lib = load()
    B, Hq, D = q.shape
    Bk, Hkv, S_max, Dk = kcache.shape
    if Bk != B or Dk != D or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("q/cache shape mismatch")
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D):
        raise ValueError("k_new and v_new must be [B, Hkv, D]")
    for name, t in (("kcache", kcache), ("vcache", vcache), ("k_new", k_new), ("v_new", v_new)):
        if t.dtype != q.dtype:
            raise TypeError(f"{name} must have q's dtype")
    dt = _dtype_code(q)
    if o is None:
        o = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), device=q.device, dtype=torch.float32)
    need = attn_decode_workspace_size(B, Hq, S_max, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lp = _dev(lse, "lse", dtype=torch.float32) if lse is not None else None
    rc = lib.attn_decode_append(_dev(q, "q", ndim=3), _dev(kcache, "kcache", ndim=4),
                                _dev(vcache, "vcache", ndim=4), _dev(k_new, "k_new", ndim=3),
                                _dev(v_new, "v_new", ndim=3),
                                _dev(kv_lens, "kv_lens", dtype=torch.int32, ndim=1),
                                _dev(o, "o", dtype=q.dtype, ndim=3), lp, B, Hq, Hkv, S_max, D, dt,
                                float(scale), _dev(workspace, "workspace"),
                                workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "attn_decode_append")
    return o, lse


NOALLOC_SCRATCH_BYTES = 16 << 20  # ATTN_NOALLOC_SCRATCH_BYTES in include/attn.h


def attn_decode_noalloc(q, kcache, vcache, kv_lens, o, lse=None, scale=None, stream=None):
    """Decode step that allocates nothing: for callers that cannot allocate
    device memory (a host framework that owns all of it, or a real-time loop
    that cannot afford cudaMalloc's synchronisation).  The outputs `o` (like
    q) and optional `lse` (float32 [B,Hq]) must be given; the library's fixed
    16 MiB device scratch array replaces the workspace.  Calls share that
    array, so calls that may overlap on the GPU must be serialised."""
    lib = load()
    B, Hq, D = q.shape
    Bk, Hkv, S_max, Dk = kcache.shape
    if Bk != B or Dk != D or tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("q/cache shape mismatch")
    if tuple(o.shape) != tuple(q.shape):
        raise ValueError("o must have q's shape")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    lp = _dev(lse, "lse", dtype=torch.float32) if lse is not None else None
    rc = lib.attn_decode_noalloc(_dev(q, "q", ndim=3), _dev(kcache, "kcache", ndim=4),
                                 _dev(vcache, "vcache", ndim=4),
                                 _dev(kv_lens, "kv_lens", dtype=torch.int32, ndim=1),
                                 _dev(o, "o", dtype=q.dtype, ndim=3), lp, B, Hq, Hkv, S_max, D,
                                 _dtype_code(q), float(scale), _stream(stream))
    _check(rc, "attn_decode_noalloc")
    return o, lse


def kv_cache_append(kcache, vcache, k_new, v_new, pos, dev_status=None, stream=None):
    """Write k_new/v_new [B,Hkv,D] at row pos[b] of the caches [B,Hkv,S_max,D]."""
    lib = load()
    B, Hkv, S_max, D = kcache.shape
    if tuple(vcache.shape) != tuple(kcache.shape):
        raise ValueError("cache shape mismatch")
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D):
        raise ValueError("k_new/v_new must be [B,Hkv,D]")
    for t in (vcache, k_new, v_new):
        if t.dtype != kcache.dtype:
            raise TypeError("cache and new rows must share one dtype")
    ds = _dev(dev_status, "dev_status", dtype=torch.int32) if dev_status is not None else None
    rc = lib.kv_cache_append(_dev(kcache, "kcache"), _dev(vcache, "vcache"),
                             _dev(k_new, "k_new"), _dev(v_new, "v_new"),
                             _dev(pos, "pos", dtype=torch.int32, ndim=1), B, Hkv, S_max, D,
                             _dtype_code(kcache), ds, _stream(stream))
    _check(rc, "kv_cache_append")


def attn_kernel_launches() -> int:
    return int(load().attn_kernel_launches())


ATTN_SELFTEST_ERROR = 0x1EE  # 0x100 (wait timed out) | site 0xEE


def attn_selftest_wait_timeout(stream=None) -> None:
    """Launch the bounded-wait self test (see include/attn.h); the error it
    records is read with attn_device_error()."""
    _check(load().attn_selftest_wait_timeout(_stream(stream)), "attn_selftest_wait_timeout")


def attn_device_error(clear: bool = True) -> int:
    code = ctypes.c_int(0)
    _check(load().attn_device_error(ctypes.byref(code), int(bool(clear))), "attn_device_error")
    return code.value
