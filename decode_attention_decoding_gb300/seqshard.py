"""Sequence-sharded decode: each rank holds one range of cache positions.

When one request's KV cache is longer than one GPU should hold (or read), the
ranks of a process group split its positions: rank r keeps positions
[begin_r, end_r) of every request and computes, with ``fd_decode_partial``
(or ``fd_decode_paged_partial``), the attention over its own range -- an
output normalised over the range and its natural-log LSE.  One all-gather
exchanges those partials (``rows * (head_dim + 1) * 4`` bytes per rank, rows =
batch x q_len x query heads) and every rank merges them with
``fd_merge_partials`` into the whole-cache result.  This is the split-K scheme
of the Flash-Decoding section of "FlashAttention 与推理算子" (splits combined
by their softmax statistics; empty splits skipped), with the splits spread
over ranks instead of CTAs.

The exchange is plain ``torch.distributed`` (NCCL on GPUs, gloo on CPU
tensors); the arithmetic runs in the library's kernels.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import fd_decode_paged_partial, fd_decode_partial, fd_merge_partials


def all_gather_partials(o_part: torch.Tensor, lse_part: torch.Tensor, group=None):
    """Every rank's partial (o_part [..., D], lse_part [...]) stacked in rank
    order: returns (o_parts [world, ..., D], lse_parts [world, ...])."""
    world = dist.get_world_size(group)
    o_part, lse_part = o_part.contiguous(), lse_part.contiguous()
    o_list = [torch.empty_like(o_part) for _ in range(world)]
    l_list = [torch.empty_like(lse_part) for _ in range(world)]
    dist.all_gather(o_list, o_part, group=group)
    dist.all_gather(l_list, lse_part, group=group)
    return torch.stack(o_list), torch.stack(l_list)


def sharded_decode(q, k_shard, v_shard, seq_lens, kv_begin, kv_end, group=None, block_table=None, **kw):
    """Decode attention over a cache whose positions are split among the
    ranks of `group`: this rank holds positions [kv_begin, kv_end) of every
    request (contiguous k_shard/v_shard [B, S, Hkv, D] with row t' = position
    kv_begin + t', or pages behind a block table of the range's own tokens).
    seq_lens are the requests' whole lengths.  Returns (out, lse), the
    whole-cache result, on every rank."""
    if block_table is None:
        o, l = fd_decode_partial(q, k_shard, v_shard, seq_lens, kv_begin, kv_end, **kw)
    else:
        o, l = fd_decode_paged_partial(q, k_shard, v_shard, block_table, seq_lens, kv_begin, kv_end, **kw)
    o_parts, l_parts = all_gather_partials(o, l, group)
    return fd_merge_partials(o_parts, l_parts)
