"""Fused lm_head (tcgen05 GEMM with a statistics epilogue) against the float64
oracle (numpy matmul of the same bf16 hidden and W, then the plain
definitions).  Tolerance: 5e-3 absolute on logprob and entropy (bf16 operands,
fp32 accumulation in tensor memory)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import lmhead as olm
from helpers import to_oracle

pytestmark = pytest.mark.gpu
IGN = -100
TOL = 5e-3


def _draw(T, V, d, w_std, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    h = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    W = (w_std * torch.randn(V, d, generator=g, device="cuda")).to(torch.bfloat16)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    return h, W, y


def _close(lp, ent, ref, rows=None):
    a = lp.double().cpu().numpy()
    e = ent.double().cpu().numpy()
    if rows is not None:
        a, e = a[rows], e[rows]
    assert np.max(np.abs(a - ref["logprob"])) <= TOL, np.max(np.abs(a - ref["logprob"]))
    assert np.max(np.abs(e - ref["entropy"])) <= TOL, np.max(np.abs(e - ref["entropy"]))


@pytest.mark.parametrize("T,V,d", [(200, 5000, 256), (128, 4096, 64), (1, 300, 128),
                                   (333, 12345, 512)])
def test_lmhead_small(cuda_lib, T, V, d):
    """Ragged token and vocabulary tails, several chunks, short and long K."""
    h, W, y = _draw(T, V, d, 0.1, T + V + d)
    y[0] = IGN
    err = cuda_lib.new_error_flag(h.device)
    lp, ent, rs = cuda_lib.lmhead_forward(h, W, y, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = olm.forward(to_oracle(h), to_oracle(W), y.cpu().numpy(), IGN)
    _close(lp, ent, ref)
    L = (rs[:, 0].double() + rs[:, 1].double()).cpu().numpy()
    assert np.max(np.abs(L - (ref["M"] + ref["logS"]))) <= TOL


def test_lmhead_matches_unfused_path(cuda_lib):
    """The fused statistics equal the unfused kernels run on fp32 logits
    formed by an fp32 matmul of the same operands."""
    T, V, d = 512, 20000, 1024
    h, W, y = _draw(T, V, d, 0.05, 7)
    lp, ent, rs = cuda_lib.lmhead_forward(h, W, y, IGN)
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    z = h.float() @ W.float().t()
    torch.backends.cuda.matmul.allow_tf32 = prev
    lp2, ent2, rs2 = cuda_lib.forward(z, y, IGN)
    torch.cuda.synchronize()
    assert torch.max(torch.abs(lp - lp2)).item() <= 1e-3
    assert torch.max(torch.abs(ent - ent2)).item() <= 1e-3


def test_lmhead_full_config_sampled(cuda_lib):
    """hidden [16384, 4096] N(0,1), W [151936, 4096] N(0, 0.02^2), sampled labels;
    every row on the GPU, 48 sampled rows through the float64 oracle."""
    from vocab_wide_token_gb300 import inputs

    d = inputs.lmhead_workload(4, "cuda")
    h, W, y = d["hidden"], d["W"], d["labels"]
    err = cuda_lib.new_error_flag(h.device)
    lp, ent, rs = cuda_lib.lmhead_forward(h, W, y, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rng = np.random.default_rng(4)
    T = h.shape[0]
    rows = np.unique(np.concatenate([[0, 127, 128, T - 1], rng.choice(T, 44, replace=False)]))
    ref = olm.forward(to_oracle(h), to_oracle(W), y.cpu().numpy(), IGN, rows=rows)
    _close(lp, ent, ref, rows)
    # batch invariance: the probe rows alone give the same bits as in the full batch
    for r in rows[:6]:
        lp1, ent1, _ = cuda_lib.lmhead_forward(h[r:r + 1], W, y[r:r + 1], IGN)
        assert torch.equal(lp1.view(torch.int32), lp[r:r + 1].view(torch.int32)), r
        assert torch.equal(ent1.view(torch.int32), ent[r:r + 1].view(torch.int32)), r
