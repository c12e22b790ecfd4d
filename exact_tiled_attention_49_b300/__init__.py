"""Exact tiled attention for B300 (sm_103a).

O = softmax(Q K^T * scale + mask) V computed tile by tile with an online
softmax so that the score matrix never reaches HBM: a causal/padding-masked
prefill forward with per-row log-sum-exp, a split-KV single-query decode step
with GQA/MQA head sharing, and an O(1) KV-cache append.

The work is done by hand-written CUDA kernels in ``libattn.so`` behind a C
ABI (``include/attn.h``); this package is a thin ctypes binding of it.
"""
from ._lib import (ATTN_BF16, ATTN_ERR_CUDA, ATTN_F16, ATTN_ERR_INVALID_ARG,  # noqa: F401
                   ATTN_ERR_UNSUPPORTED, ATTN_ERR_WORKSPACE, ATTN_F32, ATTN_OK,
                   LIB_PATH, NOALLOC_SCRATCH_BYTES, SIGNATURES, AttnError, attn_decode,
                   attn_decode_append,
                   attn_decode_noalloc,
                   attn_bwd, attn_bwd_workspace_size,
                   attn_decode_workspace_size, attn_device_error, attn_fwd, attn_fwd_chunked,
                   attn_fwd_fp8, attn_fwd_host, attn_fwd_host_workspace_size,
                   attn_fwd_kv_shard, attn_lse_merge,
                   attn_selftest_wait_timeout, ATTN_SELFTEST_ERROR,
                   attn_kernel_launches, attn_status_string, kv_cache_append, load,
                   status_string)

__all__ = [
    "attn_fwd", "attn_fwd_host", "attn_fwd_host_workspace_size", "attn_fwd_chunked", "attn_fwd_fp8", "attn_fwd_kv_shard", "attn_lse_merge", "attn_bwd", "attn_bwd_workspace_size", "attn_decode", "attn_decode_append", "attn_decode_workspace_size", "attn_decode_noalloc",
    "kv_cache_append",
    "attn_status_string", "attn_kernel_launches", "attn_device_error", "AttnError",
    "attn_selftest_wait_timeout", "ATTN_SELFTEST_ERROR",
    "load", "LIB_PATH",
]
