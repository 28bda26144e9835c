"""Vocabulary-parallel (tensor-parallel) orchestration: each rank holds the
logits of one vocabulary shard [b_s, b_{s+1}) of every row.

The exchange is one all-gather of every rank's [T, 4] shard statistics
(M_s, S_s, U_s, z_y) -- not MAX/SUM all-reduces, whose summation order is the
collective library's -- after which every rank folds them in ascending shard
order with the same kernel and holds the same bits.  The backward needs no
communication: each rank writes its own columns from the global (M, ln S).

The statistics, the combine and the backward are the C ABI's
pstat_shard_stats, pstat_combine_shards and pstat_backward_shard (through
``pstat``); the collectives here use torch.distributed.  With NCCL the
tensors stay on the GPU; with gloo (CPU process groups) they are staged
through host memory and the results moved back to the logits' device.

``tp_forward_backward_gather`` is the path the method replaces, kept as the
comparator: every rank all-gathers the [T, V_local] logit shards into the
full [T, V] logits and runs the full-vocabulary forward and backward on them
(torchtitan PR #4685, "[RL] Avoid full-vocab gather for TP policy
statistics": the legacy trainer path redistributes the vocabulary-sharded
logits to replicated form before a plain cross entropy).
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def _staged(group) -> bool:
    """Collectives of this group run on host tensors (gloo)."""
    return dist.get_backend(group) != "nccl"


def _all_gather_rows(local: torch.Tensor, group) -> torch.Tensor:
    """[world, *local.shape]: every rank's `local` (equal shapes), in rank
    order, on local's device."""
    world = dist.get_world_size(group)
    src = local.contiguous()
    if _staged(group):
        src = src.cpu()
    full = torch.empty((world * src.shape[0],) + tuple(src.shape[1:]), dtype=src.dtype,
                       device=src.device)  # concatenated form
    dist.all_gather_into_tensor(full, src, group=group)
    return full.view((world,) + tuple(src.shape)).to(local.device)


def gather_shard_layout(vocab_start: int, width: int, group=None):
    """Every rank's (vocab_start, width), gathered in rank order; returns the
    shard bounds [b_0 = 0, ..., b_S] (rank r holds [b_r, b_{r+1})).  The ranks
    must tile the vocabulary in rank order."""
    dev = "cpu" if _staged(group) else "cuda"
    mine = torch.tensor([int(vocab_start), int(width)], dtype=torch.int64, device=dev)
    allv = _all_gather_rows(mine, group).cpu().tolist()
    bounds = [0]
    for start, w in allv:
        if start != bounds[-1] or w < 1:
            raise ValueError(f"vocabulary shards must tile [0, V) in rank order: {allv}")
        bounds.append(start + w)
    return bounds


def gather_shard_stats(local: torch.Tensor, group=None) -> torch.Tensor:
    """All-gather of this rank's [T, 4] shard statistics into [T, world, 4]
    (shard index = rank) on local's device.  An all-gather, not a reduction:
    the fold order is fixed afterwards by combine_shards."""
    if local.dim() != 2 or local.shape[1] != 4:
        raise ValueError("local shard statistics must be [T, 4]")
    return _all_gather_rows(local, group).permute(1, 0, 2).contiguous()


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


def gather_logits(logits_local: torch.Tensor, bounds, group=None) -> torch.Tensor:
    """The full [T, V] logits from every rank's [T, b_{r+1} - b_r] shard
    (shards may be uneven: each is padded to the widest before the
    all-gather and cut back after it)."""
    widths = [b1 - b0 for b0, b1 in zip(bounds[:-1], bounds[1:])]
    T, w = logits_local.shape
    wmax = max(widths)
    padded = logits_local
    if w < wmax:
        padded = torch.zeros(T, wmax, dtype=logits_local.dtype, device=logits_local.device)
        padded[:, :w] = logits_local
    parts = _all_gather_rows(padded, group)  # [world, T, wmax]
    return torch.cat([parts[r, :, :widths[r]] for r in range(len(widths))], dim=1)


def tp_forward_backward_gather(logits_local: torch.Tensor, labels: torch.Tensor | None,
                               weights: torch.Tensor | None, vocab_start: int,
                               ignore_index: int = -100, out_dtype: torch.dtype | None = None,
                               group=None, *, dev_error=None):
    """The full-gather comparator: all-gather the logit shards into [T, V],
    run the full-vocabulary forward and backward on them, and keep this
    rank's columns of dlogits.  Returns (logprob, entropy, rowstats,
    dlogits_local, shard_bounds)."""
    from . import pstat

    bounds = gather_shard_layout(vocab_start, logits_local.shape[1], group)
    full = gather_logits(logits_local, bounds, group)
    lp, ent, rs, g = pstat.forward_backward(full, labels, weights, ignore_index, None, out_dtype,
                                            dev_error=dev_error)
    rank = bounds.index(vocab_start)
    return lp, ent, rs, g[:, bounds[rank]:bounds[rank + 1]], bounds


class TPPolicyStats(torch.autograd.Function):
    """Vocabulary-parallel logprob (differentiable in this rank's logits) and
    entropy (a no-grad metric): tp_forward, then in the backward this rank's
    columns of grad_logprob_t (onehot(y_t) - softmax(z_t)) through tp_backward,
    with no communication."""

    @staticmethod
    def forward(ctx, logits_local, labels, vocab_start, ignore_index=-100, group=None):
        lp, ent, rs, bounds = tp_forward(logits_local, labels, vocab_start, ignore_index, group)
        ctx.save_for_backward(logits_local, labels, rs)
        ctx.vocab_start = int(vocab_start)
        ctx.vocab_total = int(bounds[-1])
        ctx.ignore_index = ignore_index
        ctx.mark_non_differentiable(ent)
        return lp, ent

    @staticmethod
    def backward(ctx, grad_lp, grad_ent):
        logits_local, labels, rs = ctx.saved_tensors
        g = tp_backward(logits_local, labels, grad_lp.float().contiguous(), rs, ctx.vocab_start,
                        ctx.vocab_total, ctx.ignore_index)
        return g, None, None, None, None


def tp_policy_stats(logits_local: torch.Tensor, labels: torch.Tensor | None, vocab_start: int,
                    ignore_index: int = -100, group=None):
    """Differentiable (logprob, entropy) of the vocabulary-sharded logits:
    every rank gets the same bits, and each rank's gradient is its columns."""
    return TPPolicyStats.apply(logits_local, labels, vocab_start, ignore_index, group)
