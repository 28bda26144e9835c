"""Vocabulary-parallel (tensor-parallel) orchestration: each rank holds the
logits of one vocabulary shard [b_s, b_{s+1}) of every row.

The exchange is one all-gather of every rank's [T, 4] shard statistics
(M_s, S_s, U_s, z_y) -- not MAX/SUM all-reduces, whose summation order is the
collective library's -- after which every rank folds them in ascending shard
order with the same kernel and holds the same bits.  The backward needs no
communication: each rank writes its own columns from the global (M, ln S).

The statistics, the combine and the backward are the C ABI's
pstat_shard_stats, pstat_combine_shards and pstat_backward_shard (through
``pstat``); the collectives here use torch.distributed (NCCL on GPUs; the
gather helpers also run on gloo with CPU tensors).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def gather_shard_layout(vocab_start: int, width: int, group=None):
    """Every rank's (vocab_start, width), gathered in rank order; returns the
    shard bounds [b_0 = 0, ..., b_S] (rank r holds [b_r, b_{r+1})).  The ranks
    must tile the vocabulary in rank order."""
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    mine = torch.tensor([int(vocab_start), int(width)], dtype=torch.int64, device=dev)
    world = dist.get_world_size(group)
    allv = torch.empty(world * 2, dtype=torch.int64, device=dev)  # concatenated form
    dist.all_gather_into_tensor(allv, mine, group=group)
    allv = allv.view(world, 2).cpu().tolist()
    bounds = [0]
    for start, w in allv:
        if start != bounds[-1] or w < 1:
            raise ValueError(f"vocabulary shards must tile [0, V) in rank order: {allv}")
        bounds.append(start + w)
    return bounds


def gather_shard_stats(local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of this rank's [T, 4] shard statistics into [T, world, 4]
    (shard index = rank).  An all-gather, not a reduction: the fold order is
    fixed afterwards by combine_shards."""
    if local.dim() != 2 or local.shape[1] != 4:
        raise ValueError("local shard statistics must be [T, 4]")
    world = dist.get_world_size(group)
    T = local.shape[0]
    full = torch.empty(world * T, 4, dtype=local.dtype, device=local.device)  # concatenated form
    dist.all_gather_into_tensor(full, local.contiguous(), group=group)
    return full.view(world, T, 4).permute(1, 0, 2).contiguous()


def tp_forward(logits_local: torch.Tensor, labels: torch.Tensor | None, vocab_start: int,
               ignore_index: int = -100, group=None, *, dev_error=None):
    """Vocabulary-parallel forward: this rank's shard statistics, one
    all-gather of [T, 4] per rank, then the fixed-order combine.  Returns
    (logprob, entropy, rowstats, shard_bounds), the same bits on every rank."""
    from . import pstat

    bounds = gather_shard_layout(vocab_start, logits_local.shape[1], group)
    local = pstat.shard_stats(logits_local, labels, vocab_start, ignore_index, dev_error=dev_error)
    gathered = gather_shard_stats(local, group)
    lp, ent, rs = pstat.combine_shards(gathered, labels, bounds, ignore_index, dev_error=dev_error)
    return lp, ent, rs, bounds


def tp_backward(logits_local: torch.Tensor, labels: torch.Tensor | None,
                weights: torch.Tensor | None, rowstats: torch.Tensor, vocab_start: int,
                vocab_total: int, ignore_index: int = -100,
                out_dtype: torch.dtype | None = None, *, dev_error=None):
    """Vocabulary-parallel backward: this rank's columns of dlogits from the
    global (M, ln S); no communication."""
    from . import pstat

    return pstat.backward_shard(logits_local, labels, weights, rowstats, vocab_start,
                                vocab_total, ignore_index, out_dtype, dev_error=dev_error)
