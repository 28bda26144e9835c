"""Full-size workloads (V = 151,936) in the launch configuration the benchmark
times, checked against the float64 oracle on EVERY row: logprob and entropy
of all rows, and dlogits of all rows element by element (the oracle's rows
are produced in blocks of 256 and compared on the GPU with the same rule as
the small tests).  Properties that hold at any size (the gradient's zero sum,
exactly zero rows) are checked as well."""
import numpy as np
import pytest
import torch

import oracle
from helpers import GradParity, assert_forward_close, to_oracle

pytestmark = pytest.mark.gpu
IGN = -100
BLOCK = 256


def _sum_bound(w, out_dtype):
    # Sum over the vocabulary of w (onehot - p) is 0.  Each element carries
    # at most half an ulp of output rounding; sum |g| <= 2 |w|.
    w = np.abs(w)
    return (2.0**-8 if out_dtype == torch.bfloat16 else 4e-6) * w * 1.001 + 1e-7


def _grad_all_rows(grads, zo, yo, wo, out_dtype, what):
    """Every row of each tensor in `grads` ([(name, [T, V] tensor)]) against
    the oracle's dlogits, in blocks of BLOCK rows."""
    checks = [GradParity(out_dtype, f"{what} {name}") for name, _ in grads]
    T = zo.shape[0]
    for r0 in range(0, T, BLOCK):
        r1 = min(T, r0 + BLOCK)
        gref = oracle.backward(zo[r0:r1], yo[r0:r1], wo[r0:r1], IGN)
        for chk, (_, g) in zip(checks, grads):
            chk.add(g[r0:r1], gref, r0)
    for chk in checks:
        assert chk.finish() == T


@pytest.fixture(scope="module")
def fwd_data():
    from vocab_wide_token_gb300 import inputs
    return inputs.forward_workload(1, "cuda")


def test_forward_config(cuda_lib, fwd_data):
    """T=4096 bf16 N(0, 2^2), 10% peaked rows, sampled labels: every row."""
    z, y = fwd_data["logits"], fwd_data["labels"]
    err = cuda_lib.new_error_flag(z.device)
    lp, ent, rs = cuda_lib.forward(z, y, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle.forward(to_oracle(z), y.cpu().numpy(), IGN)
    assert_forward_close(lp, ent, ref, z.dtype, what="forward")
    # the row statistics too: M exactly (a maximum), ln S to the same rule
    M = rs[:, 0].double().cpu().numpy()
    assert np.array_equal(M, ref["M"])
    lnS = rs[:, 1].double().cpu().numpy()
    assert np.max(np.abs(lnS - ref["logS"])) <= 1e-4
    assert torch.all(torch.isfinite(lp)) and torch.all(ent > 0)


@pytest.fixture(scope="module")
def fb_data():
    from vocab_wide_token_gb300 import inputs
    return inputs.fwdbwd_workload(2, "cuda")


def test_fwdbwd_config(cuda_lib, fb_data):
    """T=8192 bf16, sampled labels, weights N(0,1) x mask (20% zero), bf16
    dlogits: the two calls and the single pass, every row and element."""
    z, y, w = fb_data["logits"], fb_data["labels"], fb_data["weights"]
    err = cuda_lib.new_error_flag(z.device)
    lp, ent, rs = cuda_lib.forward(z, y, IGN, dev_error=err)
    g = cuda_lib.backward(z, y, w, rs, IGN, dev_error=err)
    lp2, ent2, rs2, g2 = cuda_lib.forward_backward(z, y, w, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    zo = to_oracle(z)
    yo = y.cpu().numpy()
    wo = w.double().cpu().numpy()
    ref = oracle.forward(zo, yo, IGN)
    assert_forward_close(lp, ent, ref, z.dtype, what="fwdbwd two calls")
    assert_forward_close(lp2, ent2, ref, z.dtype, what="fwdbwd single pass")
    _grad_all_rows([("two calls", g), ("single pass", g2)], zo, yo, wo, torch.bfloat16, "fwdbwd")
    # every row: the gradient sums to zero within the output rounding bound
    s = g.double().sum(dim=1).cpu().numpy()
    bound = _sum_bound(wo, torch.bfloat16)
    assert np.all(np.abs(s) <= bound), float(np.max(np.abs(s) - bound))
    # zero-weight rows are exactly zero
    zero = (w == 0)
    assert torch.all(g[zero] == 0) and torch.all(g2[zero] == 0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_uneven_shards_config(cuda_lib, dtype):
    """T=8192, shards 50000/50000/51936, 25% rows with 10% of columns at -inf,
    5% ignored labels: sharded vs full vocabulary vs oracle on every row;
    dlogits of every row in bf16 and, for fp32 logits, in fp32; repeat run
    bitwise."""
    from vocab_wide_token_gb300 import inputs

    d = inputs.uneven_workload(3, "cuda", dtype=dtype)
    z, y, b = d["logits"], d["labels"], d["shard_bounds"]
    w = torch.randn(z.shape[0], device="cuda",
                    generator=torch.Generator(device="cuda").manual_seed(33))
    err = cuda_lib.new_error_flag(z.device)
    lp_s, ent_s, rs_s = cuda_lib.forward(z, y, IGN, b, dev_error=err)
    lp_f, ent_f, rs_f = cuda_lib.forward(z, y, IGN, None, dev_error=err)
    lp_s2, ent_s2, _ = cuda_lib.forward(z, y, IGN, b)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(lp_s.view(torch.int32), lp_s2.view(torch.int32))
    assert torch.equal(ent_s.view(torch.int32), ent_s2.view(torch.int32))
    zo = to_oracle(z)
    yo = y.cpu().numpy()
    wo = w.double().cpu().numpy()
    ref = oracle.sharded(zo, yo, b, IGN)
    assert_forward_close(lp_s, ent_s, ref, dtype, what="uneven sharded")
    assert_forward_close(lp_f, ent_f, ref, dtype, what="uneven full vocabulary")
    outs = [torch.bfloat16] + ([torch.float32] if dtype == torch.float32 else [])
    for out_dtype in outs:
        g = cuda_lib.backward(z, y, w, rs_s, IGN, out_dtype=out_dtype, dev_error=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        _grad_all_rows([("sharded", g)], zo, yo, wo, out_dtype, f"uneven {dtype} -> {out_dtype}")
        # masked columns carry exactly zero gradient
        mrow = int(d["masked_rows"][0])
        assert torch.all(g[mrow][torch.isinf(z[mrow].float())] == 0)
        del g
