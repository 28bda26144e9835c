"""The vocabulary-parallel path across processes, with the real kernels: two
gloo ranks (separate processes, both on the one GPU) each hold one uneven
vocabulary shard of the same logits.  Each runs pstat_shard_stats on its
shard, all-gathers the [T, 4] statistics through the process group, folds
them with pstat_combine_shards and writes its columns with
pstat_backward_shard; each also runs the full-gather comparator (all-gather
of the logit shards, then the full-vocabulary single pass).

Checked against single-process calls on the whole logits:
  - sharded path: logprob, entropy, (M, ln S) bit for bit equal to
    pstat_forward with the same shard bounds, on both ranks; each rank's
    dlogits columns bit for bit equal to those of pstat_backward;
  - full-gather path: bit for bit equal to pstat_forward_backward on the
    whole logits ({0, V});
  - both paths against the float64 oracle within the parity tolerances
    (sharded and full-vocabulary sums agree to rounding, not bitwise).
The ranks never wait on one another inside a kernel: the exchange is a host
collective between kernel launches."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from helpers import assert_forward_close, assert_grad_close, to_oracle

pytestmark = pytest.mark.gpu
IGN = -100


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _draw(T, V, dtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    z = 2.0 * torch.randn(T, V, generator=g, device="cuda")
    z[5, : V // 4] = -math.inf
    z = z.to(dtype)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    y[3] = IGN
    w = torch.randn(T, generator=g, device="cuda")
    w[4] = 0.0
    return z, y, w


def _rank(rank, world, port, T, V, bounds, dtype_name, seed, outdir):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from vocab_wide_token_gb300 import pstat, tp

        torch.cuda.set_device(0)
        z, y, w = _draw(T, V, getattr(torch, dtype_name), seed)
        b0, b1 = bounds[rank], bounds[rank + 1]
        zl = z[:, b0:b1].contiguous()
        err = pstat.new_error_flag(z.device)
        lp, ent, rs, got_bounds = tp.tp_forward(zl, y, b0, IGN, dev_error=err)
        g = tp.tp_backward(zl, y, w, rs, b0, V, IGN, dev_error=err)
        lpG, entG, rsG, gG, _ = tp.tp_forward_backward_gather(zl, y, w, b0, IGN, dev_error=err)
        # autograd: d sum(w logprob) / d logits is this rank's columns of the
        # weighted backward with weights w
        zA = zl.detach().clone().requires_grad_(True)
        lpA, _ = tp.tp_policy_stats(zA, y, b0, IGN)
        (lpA * w).sum().backward()
        torch.cuda.synchronize()
        torch.save({"bounds": got_bounds, "err": int(err.item()), "lp": lp.cpu(),
                    "ent": ent.cpu(), "rs": rs.cpu(), "g": g.cpu(), "lpG": lpG.cpu(),
                    "entG": entG.cpu(), "rsG": rsG.cpu(), "gG": gG.contiguous().cpu(),
                    "lpA": lpA.detach().cpu(), "gA": zA.grad.cpu()},
                   os.path.join(outdir, f"rank{rank}.pt"))
    finally:
        dist.destroy_process_group()


def _bits(x):
    x = x.contiguous()
    return x.view(torch.int16 if x.element_size() == 2 else torch.int32)


@pytest.mark.parametrize("dtype,T,V,bounds", [
    (torch.bfloat16, 256, 151936, [0, 50000, 151936]),
    (torch.float32, 200, 10007, [0, 4001, 10007]),
])
def test_two_ranks_real_kernels(cuda_lib, tmp_path, dtype, T, V, bounds):
    world = 2
    seed = V + T
    mp.start_processes(_rank, args=(world, _free_port(), T, V, bounds, str(dtype).split(".")[1],
                                    seed, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    z, y, w = _draw(T, V, dtype, seed)
    lp, ent, rs = cuda_lib.forward(z, y, IGN, bounds)
    gfull = cuda_lib.backward(z, y, w, rs, IGN)
    lpF, entF, rsF, gF = cuda_lib.forward_backward(z, y, w, IGN)
    torch.cuda.synchronize()
    zo, yo = to_oracle(z), y.cpu().numpy()
    ref = oracle.forward(zo, yo, IGN)
    rows = np.array([0, 1, 3, 4, 5, 77, T - 1])
    gref = oracle.backward(zo[rows], yo[rows], w[rows].double().cpu().numpy(), IGN)
    for r in range(world):
        res = torch.load(os.path.join(tmp_path, f"rank{r}.pt"))
        assert res["bounds"] == bounds and res["err"] == 0
        b0, b1 = bounds[r], bounds[r + 1]
        # sharded path == the single-process sharded forward, bit for bit
        for key, want in (("lp", lp), ("ent", ent), ("rs", rs)):
            assert torch.equal(_bits(res[key]), _bits(want.cpu())), (r, key)
        assert torch.equal(_bits(res["g"]), _bits(gfull[:, b0:b1].cpu())), r
        # the autograd function over the same path
        assert torch.equal(_bits(res["lpA"]), _bits(lp.cpu())), r
        assert torch.equal(_bits(res["gA"]), _bits(gfull[:, b0:b1].cpu())), r
        # full-gather path == the single-process full-vocabulary single pass
        for key, want in (("lpG", lpF), ("entG", entF), ("rsG", rsF)):
            assert torch.equal(_bits(res[key]), _bits(want.cpu())), (r, key)
        assert torch.equal(_bits(res["gG"]), _bits(gF[:, b0:b1].cpu())), r
        # both against the oracle
        assert_forward_close(res["lp"], res["ent"], ref, dtype, what=f"rank {r} sharded")
        assert_forward_close(res["lpG"], res["entG"], ref, dtype, what=f"rank {r} gathered")
        assert_grad_close(res["g"][rows], gref[:, b0:b1], dtype, f"rank {r} sharded")
        assert_grad_close(res["gG"][rows], gref[:, b0:b1], dtype, f"rank {r} gathered")


def _nccl_rank(index, port, T, V, seed, outdir):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), NCCL_NVLS_ENABLE="0")
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    try:
        from vocab_wide_token_gb300 import pstat, tp

        z, y, w = _draw(T, V, torch.bfloat16, seed)
        err = pstat.new_error_flag(z.device)
        lp, ent, rs, bounds = tp.tp_forward(z, y, 0, IGN, dev_error=err)
        g = tp.tp_backward(z, y, w, rs, 0, V, IGN, dev_error=err)
        lpG, entG, rsG, gG, _ = tp.tp_forward_backward_gather(z, y, w, 0, IGN, dev_error=err)
        torch.cuda.synchronize()
        torch.save({"bounds": bounds, "err": int(err.item()), "lp": lp.cpu(), "ent": ent.cpu(),
                    "rs": rs.cpu(), "g": g.cpu(), "lpG": lpG.cpu(), "gG": gG.contiguous().cpu(),
                    "on_device": bool(lp.is_cuda and g.is_cuda)},
                   os.path.join(outdir, "nccl.pt"))
    finally:
        dist.destroy_process_group()


def test_nccl_branch_single_rank(cuda_lib, tmp_path):
    """The NCCL branch of the orchestration (collectives on device tensors,
    no host staging), exercised with one rank holding the whole vocabulary:
    the results equal the single-process calls bit for bit."""
    import torch.distributed as dist

    if not dist.is_nccl_available():
        pytest.skip("NCCL not available")
    T, V, seed = 96, 20011, 5
    mp.start_processes(_nccl_rank, args=(_free_port(), T, V, seed, str(tmp_path)), nprocs=1,
                       join=True, start_method="spawn")
    res = torch.load(os.path.join(tmp_path, "nccl.pt"))
    assert res["bounds"] == [0, V] and res["err"] == 0 and res["on_device"]
    z, y, w = _draw(T, V, torch.bfloat16, seed)
    lp, ent, rs = cuda_lib.forward(z, y, IGN)
    g = cuda_lib.backward(z, y, w, rs, IGN)
    lpF, entF, rsF, gF = cuda_lib.forward_backward(z, y, w, IGN)
    torch.cuda.synchronize()
    for key, want in (("lp", lp), ("ent", ent), ("rs", rs), ("g", g), ("lpG", lpF), ("gG", gF)):
        assert torch.equal(_bits(res[key]), _bits(want.cpu())), key
