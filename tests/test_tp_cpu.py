"""Vocabulary-parallel plumbing on CPU: two gloo ranks each hold one shard of
the vocabulary.  The layout gather returns the shard bounds in rank order and
refuses shards that do not tile the vocabulary; the statistics gather is an
all-gather that puts rank r's [T, 4] at [:, r, :]; the logit gather of the
full-gather comparator rebuilds [T, V] from uneven shards.  No GPU is
involved (the kernels that fill and fold the statistics run in the GPU
tests, with real shard statistics in tests/test_gpu_tp_ranks.py)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from vocab_wide_token_gb300 import tp

        widths = [7, 5]
        start = sum(widths[:rank])
        bounds = tp.gather_shard_layout(start, widths[rank])
        local = torch.arange(3 * 4, dtype=torch.float32).reshape(3, 4) + 100 * rank
        gathered = tp.gather_shard_stats(local)
        full = torch.arange(3 * 12, dtype=torch.float32).reshape(3, 12)
        logits = tp.gather_logits(full[:, start:start + widths[rank]].clone(), bounds)
        try:
            tp.gather_shard_layout(0, 4)  # both ranks claim the first columns
            overlap_refused = False
        except ValueError:
            overlap_refused = True
        out[rank] = (bounds, gathered.tolist(), logits.tolist(), overlap_refused)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_gather_shards():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    base = torch.arange(12, dtype=torch.float32).reshape(3, 4)
    want = torch.stack([base, base + 100], dim=1)  # [T, rank, 4]
    full = torch.arange(3 * 12, dtype=torch.float32).reshape(3, 12)
    for r in range(world):
        bounds, gathered, logits, refused = res[r]
        assert bounds == [0, 7, 12]
        assert torch.equal(torch.tensor(gathered), want)
        assert torch.equal(torch.tensor(logits), full)
        assert refused
