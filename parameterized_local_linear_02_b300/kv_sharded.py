"""Decode with every sequence's key range sharded over the ranks of a process
group: rank r holds cache positions key_begin_r .. key_begin_r + S_r - 1 of
every sequence, computes the online-softmax states of its slice
(plx_decode_partials), the ranks exchange them (one all-gather of
B*H*splits*(2d+4) fp32 values per rank), and each rank merges all of them
with the log-sum-exp combine (plx_decode_combine).  The merge of disjoint key
ranges is exact, so the result equals plx_decode over the whole range up to
fp32 rounding of the merge order ("Parallax: Parameterized Local Linear
Attention for Language Modeling", gist.science, "Algoritmo Consapevole
dell'Hardware": the decode is one pass over the K/V stream with an online
softmax, whose states merge by their log-sum-exp weights).

The host logic here is the exchange: every rank must use the same split
count (agreed by a max over the group), and the gathered buffer is rank-major,
which is the shard order the combine expects.  The arithmetic runs in the
library's CUDA kernels.
"""
from __future__ import annotations

import torch

from .binding import plx_decode_combine, plx_decode_num_splits, plx_decode_partials

__all__ = ["agree_num_splits", "gather_partials", "plx_decode_kv_sharded"]


def agree_num_splits(num_splits: int, group=None) -> int:
    """The largest split count any rank proposes (every rank must pass the
    combine the same count)."""
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend(group) == "gloo" else torch.device("cuda", torch.cuda.current_device())
    t = torch.tensor([int(num_splits)], dtype=torch.int64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return int(t.item())


def gather_partials(partials: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather every rank's flat partials buffer: [world][...] in rank
    order, returned flat (the combine's [groups][B*H][splits][2d+4])."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = torch.empty(world * partials.numel(), dtype=partials.dtype, device=partials.device)
    dist.all_gather_into_tensor(out, partials.contiguous(), group=group)
    return out


def plx_decode_kv_sharded(q, rho, k_shard, v_shard, seqlens, *, key_begin, group=None, num_splits=None,
                          scale=None, out_dtype=torch.bfloat16, with_lse=True):
    """One-token PLX decode with the K/V range sharded over ``group``.

    ``q``, ``rho`` [B, H, d] and ``seqlens`` [B] (int32) are the same on every
    rank; ``k_shard``, ``v_shard`` [B, H, S_r, d] are this rank's positions
    ``key_begin`` .. ``key_begin + S_r - 1``.  The shards must cover
    0 .. max(seqlens) - 1 without overlap.  Returns ``(out, lse)`` on every
    rank."""
    import torch.distributed as dist
    B, H, S, d = k_shard.shape
    n = num_splits if num_splits else plx_decode_num_splits(B, H, d, S)
    n = agree_num_splits(n, group)
    parts = plx_decode_partials(q, rho, k_shard, v_shard, seqlens, key_begin=key_begin, num_splits=n, scale=scale)
    allp = gather_partials(parts, group)
    return plx_decode_combine(allp, groups=dist.get_world_size(group), num_splits=n, B=B, H=H, d=d,
                              with_rho=rho is not None, out_dtype=out_dtype, with_lse=with_lse)
