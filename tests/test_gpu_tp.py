"""Vocabulary-parallel entry points on one GPU, the ranks emulated in one
process: pstat_shard_stats on every shard's columns, the [T, 4] statistics
stacked in shard order (what the all-gather produces), then
pstat_combine_shards -- bit for bit the single call pstat_forward with those
shard bounds; pstat_backward_shard on each shard -- bit for bit that shard's
columns of pstat_backward."""
import math

import pytest
import torch

import oracle
from helpers import assert_forward_close, to_oracle

pytestmark = pytest.mark.gpu
IGN = -100


def _bits(x):
    x = x.contiguous()
    return x.view(torch.int16 if x.element_size() == 2 else torch.int32)


def _emulate(pstat, z, y, bounds, err):
    parts = [pstat.shard_stats(z[:, b0:b1], y, b0, IGN, dev_error=err)
             for b0, b1 in zip(bounds[:-1], bounds[1:])]
    return pstat.combine_shards(torch.stack(parts, dim=1), y, bounds, IGN, dev_error=err)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("V,bounds", [(10007, [0, 5003, 10007]),
                                      (10007, [0, 513, 4001, 6000, 10007]),
                                      (151936, [0, 50000, 100000, 151936]),
                                      (3000, [0, 3000])])
def test_shards_equal_sharded_forward_and_backward(cuda_lib, dtype, V, bounds):
    g = torch.Generator(device="cuda").manual_seed(V + len(bounds))
    T = 200
    z = 2.0 * torch.randn(T, V, generator=g, device="cuda")
    if len(bounds) > 2:
        z[7, bounds[1]:bounds[2]] = -math.inf  # one shard fully masked
        z[8, : bounds[1]] = -math.inf
    z = z.to(dtype)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    y[3] = IGN
    y[4] = V + 5                               # outside the vocabulary
    y[5] = bounds[-2]                          # first column of the last shard
    w = torch.randn(T, generator=g, device="cuda")
    w[6] = 0.0
    e1 = cuda_lib.new_error_flag(z.device)
    e2 = cuda_lib.new_error_flag(z.device)
    lp, ent, rs = cuda_lib.forward(z, y, IGN, bounds, dev_error=e1)
    lp2, ent2, rs2 = _emulate(cuda_lib, z, y, bounds, e2)
    torch.cuda.synchronize()
    for a, b, name in ((lp, lp2, "logprob"), (ent, ent2, "entropy"), (rs, rs2, "rowstats")):
        assert torch.equal(_bits(a), _bits(b)), name
    assert e1.item() == e2.item() and e1.item() & cuda_lib.DEV_BAD_LABEL

    out_dtype = dtype
    gfull = cuda_lib.backward(z, y, w, rs, IGN, out_dtype=out_dtype, dev_error=e1)
    for b0, b1 in zip(bounds[:-1], bounds[1:]):
        gs = cuda_lib.backward_shard(z[:, b0:b1].contiguous(), y, w, rs, b0, V, IGN, out_dtype,
                                     dev_error=e2)
        torch.cuda.synchronize()
        assert torch.equal(_bits(gs), _bits(gfull[:, b0:b1])), (b0, b1)

    keep = torch.ones(T, dtype=torch.bool)
    keep[4] = False
    rows = keep.nonzero().squeeze(1)[:40]
    ref = oracle.forward(to_oracle(z[rows.cuda()]), y[rows.cuda()].cpu().numpy(), IGN)
    assert_forward_close(lp2[rows.cuda()], ent2[rows.cuda()], ref, dtype, what=f"shards V={V}")


def test_shard_entry_argument_checks(cuda_lib):
    z = torch.randn(4, 100, device="cuda")
    y = torch.zeros(4, dtype=torch.int64, device="cuda")
    st = torch.zeros(4, 2, 4, device="cuda")
    with pytest.raises(cuda_lib.PstatError):
        cuda_lib.combine_shards(st, y, [0, 60, 50])      # bounds not increasing
    with pytest.raises(cuda_lib.PstatError):
        cuda_lib.backward_shard(z, y, None, torch.zeros(4, 2, device="cuda"), 50, 120)
