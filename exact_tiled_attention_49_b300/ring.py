"""Sequence-parallel attention across ranks: key/value shards passed round a ring.

"Building a causal self-attention block from scratch in PyTorch", Extending
It: distributed attention shards Q/K/V across devices and recombines the
results.  Each rank holds its own query rows (global positions q_pos) and
one shard of every sequence's keys and values.  In N steps every shard
visits every rank: at step s rank r holds the shard that started on rank
(r - s) mod N, computes its queries' partial attention over it
(attn_fwd_kv_shard, which takes the shard's global key offset), and passes
the shard on to rank r + 1 while receiving the next one from rank r - 1 (the
transfer is posted before the compute so the two overlap).  The partials
are stored by the shard's home rank, and attn_lse_merge combines them in
that order, so the result does not depend on the ring schedule.

The exchange uses torch.distributed point-to-point calls (NCCL between
GPUs); every rank's shards must have the same shape (pad the last one: keys
at or past key_lens are never used).  The per-shard compute and the merge
are parameters so that the exchange order can be checked with gloo on the
CPU; by default they are this library's CUDA kernels.
"""
from __future__ import annotations


def ring_attention(q, k, v, q_pos, key_lens, shard_offsets, causal=True, scale=None,
                   group=None, shard_fn=None, merge_fn=None):
    """Attention of this rank's queries over the keys of all ranks.

    q [B,Hq,T,D] this rank's queries; k, v [B,Hkv,S,D] this rank's key/value
    shard; q_pos, key_lens int32 [B] global positions (see
    attn_fwd_kv_shard); shard_offsets[r] the global key position of rank r's
    shard.  Returns (o [B,Hq,T,D], lse [B,Hq,T]).
    """
    import torch
    import torch.distributed as dist

    if shard_fn is None or merge_fn is None:
        from ._lib import attn_fwd_kv_shard, attn_lse_merge
        shard_fn = shard_fn or attn_fwd_kv_shard
        merge_fn = merge_fn or attn_lse_merge
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if len(shard_offsets) != world:
        raise ValueError("one shard offset per rank")

    def peer(r):
        return dist.get_global_rank(group, r) if group is not None else r

    nxt, prv = peer((rank + 1) % world), peer((rank - 1) % world)
    B, Hq, T, D = q.shape
    o_parts = torch.empty((world, B, Hq, T, D), dtype=q.dtype, device=q.device)
    lse_parts = torch.empty((world, B, Hq, T), dtype=torch.float32, device=q.device)
    cur_k, cur_v = k.contiguous(), v.contiguous()
    for step in range(world):
        home = (rank - step) % world
        reqs, nk, nv = [], None, None
        if step + 1 < world:
            nk, nv = torch.empty_like(cur_k), torch.empty_like(cur_v)
            ops = [dist.P2POp(dist.isend, cur_k, nxt, group), dist.P2POp(dist.isend, cur_v, nxt, group),
                   dist.P2POp(dist.irecv, nk, prv, group), dist.P2POp(dist.irecv, nv, prv, group)]
            reqs = dist.batch_isend_irecv(ops)
        shard_fn(q, cur_k, cur_v, q_pos, key_lens, int(shard_offsets[home]),
                 o=o_parts[home], lse=lse_parts[home], causal=causal, scale=scale)
        for r in reqs:
            r.wait()
        if nk is not None:
            cur_k, cur_v = nk, nv
    return merge_fn(o_parts, lse_parts)
