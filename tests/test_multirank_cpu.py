"""The multi-rank benchmark path on CPU: two gloo ranks each draw their own
batch (independent token rows, no data-path collective), and the timing takes
the slowest rank through a MAX all-reduce before the whole-job rate is formed.
No GPU is involved."""
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
        import bench
        from vocab_wide_token_gb300 import inputs

        d = inputs.fwdbwd_workload(bench.rank_seed(2, rank), "cpu", T=4, V=1000)
        gathered = [torch.empty(4, 1000, dtype=torch.bfloat16) for _ in range(world)]
        dist.all_gather(gathered, d["logits"])  # test-only: compare the ranks' batches
        differ = not torch.equal(gathered[0], gathered[1])
        ms = bench.max_over_ranks(10.0 + 5.0 * rank)
        rate = bench.whole_job_rate(4, 3, world, ms)
        out[rank] = (differ, ms, rate)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    for r in range(world):
        differ, ms, rate = res[r]
        assert differ                       # each rank works on its own rows
        assert ms == 15.0                   # the slowest rank's time on every rank
        assert abs(rate - 2 * 4 * 3 / 0.015) < 1e-6
