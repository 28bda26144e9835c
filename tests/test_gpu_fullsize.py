"""Full-size workloads (V = 151,936) in the launch configuration the benchmark
times: the GPU runs every row; the oracle checks sampled rows one by one, and
properties that hold at any size are checked on every row."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_forward_close, assert_grad_close, to_oracle

pytestmark = pytest.mark.gpu
IGN = -100


def _sample_rows(T, extra, seed, must=()):
    rng = np.random.default_rng(seed)
    rows = set([0, 1, T // 2, T - 1, *must])
    rows.update(rng.choice(T, size=extra, replace=False).tolist())
    return np.array(sorted(rows))


def _sum_bound(w, out_dtype):
    # Sum over the vocabulary of w (onehot - p) is 0.  Each element carries
    # at most half an ulp of output rounding; sum |g| <= 2 |w|.
    w = np.abs(w)
    return (2.0**-8 if out_dtype == torch.bfloat16 else 4e-6) * w * 1.001 + 1e-7


@pytest.fixture(scope="module")
def fwd_data():
    from vocab_wide_token_gb300 import inputs
    return inputs.forward_workload(1, "cuda")


def test_forward_config(cuda_lib, fwd_data):
    """T=4096 bf16 N(0, 2^2), 10% peaked rows, sampled labels."""
    z, y = fwd_data["logits"], fwd_data["labels"]
    err = cuda_lib.new_error_flag(z.device)
    lp, ent, rs = cuda_lib.forward(z, y, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    peaked = fwd_data["peaked_rows"][:8].cpu().numpy().tolist()
    rows = _sample_rows(z.shape[0], 40, 1, peaked)
    ref = oracle.forward(to_oracle(z[rows]), y[rows].cpu().numpy(), IGN)
    assert_forward_close(lp[rows], ent[rows], ref, z.dtype, what="forward")
    assert torch.all(torch.isfinite(lp)) and torch.all(ent > 0)


@pytest.fixture(scope="module")
def fb_data():
    from vocab_wide_token_gb300 import inputs
    return inputs.fwdbwd_workload(2, "cuda")


def test_fwdbwd_config(cuda_lib, fb_data):
    """T=8192 bf16, sampled labels, weights N(0,1) x mask (20% zero), bf16 dlogits."""
    z, y, w = fb_data["logits"], fb_data["labels"], fb_data["weights"]
    err = cuda_lib.new_error_flag(z.device)
    lp, ent, rs = cuda_lib.forward(z, y, IGN, dev_error=err)
    g = cuda_lib.backward(z, y, w, rs, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rows = _sample_rows(z.shape[0], 20, 2)
    zo = to_oracle(z[rows])
    yo = y[rows].cpu().numpy()
    ref = oracle.forward(zo, yo, IGN)
    assert_forward_close(lp[rows], ent[rows], ref, z.dtype, what="fwdbwd")
    gref = oracle.backward(zo, yo, w[rows].double().cpu().numpy(), IGN)
    assert_grad_close(g[rows], gref, torch.bfloat16, "fwdbwd")
    # every row: the gradient sums to zero within the output rounding bound
    s = g.double().sum(dim=1).cpu().numpy()
    bound = _sum_bound(w.double().cpu().numpy(), torch.bfloat16)
    assert np.all(np.abs(s) <= bound), float(np.max(np.abs(s) - bound))
    # zero-weight rows are exactly zero
    zero = (w == 0)
    assert torch.all(g[zero] == 0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_uneven_shards_config(cuda_lib, dtype):
    """T=8192, shards 50000/50000/51936, 25% rows with 10% of columns at -inf,
    5% ignored labels: sharded vs full vocabulary vs oracle; repeat run bitwise."""
    from vocab_wide_token_gb300 import inputs

    d = inputs.uneven_workload(3, "cuda", dtype=dtype)
    z, y, b = d["logits"], d["labels"], d["shard_bounds"]
    w = torch.randn(z.shape[0], device="cuda", generator=torch.Generator(device="cuda").manual_seed(33))
    err = cuda_lib.new_error_flag(z.device)
    lp_s, ent_s, rs_s = cuda_lib.forward(z, y, IGN, b, dev_error=err)
    lp_f, ent_f, rs_f = cuda_lib.forward(z, y, IGN, None, dev_error=err)
    out_dtype = torch.bfloat16
    g = cuda_lib.backward(z, y, w, rs_s, IGN, out_dtype=out_dtype, dev_error=err)
    lp_s2, ent_s2, _ = cuda_lib.forward(z, y, IGN, b)
    torch.cuda.synchronize()
    assert err.item() == 0
    tol = 1e-5 if dtype == torch.float32 else 1e-4
    fin = torch.isfinite(lp_f)
    assert torch.allclose(lp_s[fin], lp_f[fin], rtol=0, atol=tol)
    assert torch.allclose(ent_s, ent_f, rtol=0, atol=tol)
    assert torch.equal(lp_s.view(torch.int32), lp_s2.view(torch.int32))
    assert torch.equal(ent_s.view(torch.int32), ent_s2.view(torch.int32))
    masked = d["masked_rows"][:6].cpu().numpy().tolist()
    ign = torch.nonzero(y == IGN)[:3, 0].cpu().numpy().tolist()
    rows = _sample_rows(z.shape[0], 16, 3, masked + ign)
    zo = to_oracle(z[rows])
    yo = y[rows].cpu().numpy()
    ref = oracle.sharded(zo, yo, b, IGN)
    assert_forward_close(lp_s[rows], ent_s[rows], ref, dtype, what="uneven sharded")
    gref = oracle.backward(zo, yo, w[rows].double().cpu().numpy(), IGN)
    assert_grad_close(g[rows], gref, out_dtype, "uneven")
    # masked columns carry exactly zero gradient
    mrow = masked[0]
    assert torch.all(g[mrow][torch.isinf(z[mrow].float())] == 0)
