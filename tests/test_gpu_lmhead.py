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
                                   (333, 12345, 512), (257, 9000, 192), (300, 40000, 128),
                                   (97, 65600, 64)])
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


def _frob_rel(a, ref):
    a = np.asarray(a, np.float64)
    return float(np.linalg.norm(a - ref) / max(np.linalg.norm(ref), 1e-300))


@pytest.mark.parametrize("T,V,d", [(200, 5000, 256), (128, 4096, 64), (1, 300, 128),
                                   (333, 12345, 512), (257, 9000, 192), (300, 40000, 128),
                                   (97, 65600, 64)])
def test_lmhead_backward_small(cuda_lib, T, V, d):
    """dhidden += g W and dW += g^T hidden against float64 numpy; Frobenius-
    relative <= 1e-3 per tensor; a second call accumulates.  V = 40000 and
    65600 span two and three 32768-column chunks of the backward, the last
    one ragged (7232 columns) or narrower than a tile (64 columns)."""
    h, W, y = _draw(T, V, d, 0.1, 3 * T + V + d)
    g = torch.Generator(device="cuda").manual_seed(T + d)
    w = torch.randn(T, generator=g, device="cuda")
    if T > 3:
        y[1] = IGN
        w[2] = 0.0
    err = cuda_lib.new_error_flag(h.device)
    lp, ent, rs = cuda_lib.lmhead_forward(h, W, y, IGN, dev_error=err)
    dh, dW = cuda_lib.lmhead_backward(h, W, y, w, rs, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rdh, rdW = olm.backward(to_oracle(h), to_oracle(W), y.cpu().numpy(), w.double().cpu().numpy(), IGN)
    e1 = _frob_rel(dh.double().cpu().numpy(), rdh)
    e2 = _frob_rel(dW.double().cpu().numpy(), rdW)
    assert e1 <= 1e-3 and e2 <= 1e-3, (e1, e2)
    # accumulation: a second call adds the same gradient again
    cuda_lib.lmhead_backward(h, W, y, w, rs, IGN, dhidden=dh, dW=dW)
    torch.cuda.synchronize()
    assert _frob_rel(dh.double().cpu().numpy(), 2 * rdh) <= 1e-3
    assert _frob_rel(dW.double().cpu().numpy(), 2 * rdW) <= 1e-3


def test_lmhead_autograd(cuda_lib):
    """lmhead_policy_stats: the logprob of lmhead_forward, and grads of
    sum(c logprob) equal to lmhead_backward with weights c, cast to the
    inputs' dtype, bit for bit; entropy carries no gradient."""
    T, V, d = 200, 5000, 256
    h, W, y = _draw(T, V, d, 0.1, 11)
    y[0] = IGN
    c = torch.randn(T, generator=torch.Generator(device="cuda").manual_seed(3), device="cuda")
    lp, ent, rs = cuda_lib.lmhead_forward(h, W, y, IGN)
    dh, dW = cuda_lib.lmhead_backward(h, W, y, c, rs, IGN)
    hA = h.detach().clone().requires_grad_(True)
    WA = W.detach().clone().requires_grad_(True)
    lpA, entA = cuda_lib.lmhead_policy_stats(hA, WA, y, IGN)
    assert not entA.requires_grad
    (lpA * c).sum().backward()
    torch.cuda.synchronize()
    assert torch.equal(lpA.detach(), lp) and torch.equal(entA, ent)
    assert hA.grad.dtype == h.dtype and WA.grad.dtype == W.dtype
    assert torch.equal(hA.grad, dh.to(h.dtype)) and torch.equal(WA.grad, dW.to(W.dtype))


def _row_errors(a, ref):
    """Per row: Frobenius-relative error and max-abs error over the row's
    max-abs reference value."""
    a = np.asarray(a, np.float64)
    fro = np.linalg.norm(a - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-300)
    mx = np.max(np.abs(a - ref), axis=1) / np.maximum(np.max(np.abs(ref), axis=1), 1e-300)
    return fro, mx


@pytest.mark.parametrize("T", [256, 1024])
def test_lmhead_backward_full_vocab(cuda_lib, T):
    """T tokens against the full vocabulary and hidden size (V = 151936,
    d = 4096): every element of dhidden and dW through the float64 oracle,
    Frobenius-relative <= 1e-3 per tensor.  Beside the whole-tensor bound,
    a per-row diagnostic on 64 sampled vocabulary rows of dW (and the rows of
    eight labels) and 64 token rows of dhidden: each row within 1e-3
    Frobenius-relative on its own, and its largest element error within 2e-3
    of its largest reference element (a maximum over 4096 elements, each a
    sum carrying two fp16 roundings of 2^-12), so that one bad tile cannot
    hide in the norm of the whole tensor.  Most of a row's gradient entries
    are softmax probabilities far below 2^-14; they must keep their relative
    precision too."""
    from vocab_wide_token_gb300 import inputs

    d = inputs.lmhead_workload(5, "cuda", T=T)
    h, W, y, w = d["hidden"], d["W"], d["labels"], d["weights"]
    y[3] = IGN
    err = cuda_lib.new_error_flag(h.device)
    lp, ent, rs = cuda_lib.lmhead_forward(h, W, y, IGN, dev_error=err)
    dh, dW = cuda_lib.lmhead_backward(h, W, y, w, rs, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    rdh, rdW = olm.backward(to_oracle(h), to_oracle(W), y.cpu().numpy(), w.double().cpu().numpy(), IGN)
    dhn = dh.double().cpu().numpy()
    e1 = _frob_rel(dhn, rdh)
    rng = np.random.default_rng(T)
    V = W.shape[0]
    vrows = np.unique(np.concatenate([rng.choice(V, 64, replace=False),
                                      y[y != IGN][:8].cpu().numpy()]))
    dWs = dW[torch.from_numpy(vrows).cuda()].double().cpu().numpy()
    e2 = _frob_rel(dW.double().cpu().numpy(), rdW)
    assert e1 <= 1e-3 and e2 <= 1e-3, (e1, e2)
    fro_v, max_v = _row_errors(dWs, rdW[vrows])
    assert fro_v.max() <= 1e-3 and max_v.max() <= 2e-3, (
        f"dW rows: worst Frobenius-relative {fro_v.max():.2e} (row {vrows[fro_v.argmax()]}), "
        f"worst max-relative {max_v.max():.2e} (row {vrows[max_v.argmax()]})")
    trows = np.setdiff1d(rng.choice(T, min(64, T), replace=False), [3])
    fro_t, max_t = _row_errors(dhn[trows], rdh[trows])
    assert fro_t.max() <= 1e-3 and max_t.max() <= 2e-3, (
        f"dhidden rows: worst Frobenius-relative {fro_t.max():.2e}, max-relative {max_t.max():.2e}")
    assert np.all(dhn[3] == 0)  # the ignored token contributes nothing


def test_lmhead_backward_dhidden_batch_invariant(cuda_lib):
    """A token's dhidden row depends on that token alone (its gradient row is
    formed and scaled per row; the vocabulary chunks are accumulated in a
    fixed order), so it is bit-identical computed alone, in a sub-batch and in
    the whole batch."""
    T, V, d = 300, 20000, 512
    h, W, y = _draw(T, V, d, 0.05, 21)
    w = torch.randn(T, generator=torch.Generator(device="cuda").manual_seed(22), device="cuda")
    lp, ent, rs = cuda_lib.lmhead_forward(h, W, y, IGN)
    dh, _ = cuda_lib.lmhead_backward(h, W, y, w, rs, IGN)
    for r0, r1 in ((0, 1), (131, 132), (299, 300), (100, 229)):
        dh1, _ = cuda_lib.lmhead_backward(h[r0:r1], W, y[r0:r1], w[r0:r1], rs[r0:r1], IGN)
        torch.cuda.synchronize()
        assert torch.equal(dh1.view(torch.int32), dh[r0:r1].view(torch.int32)), (r0, r1)


def test_lmhead_backward_full_config(cuda_lib):
    """hidden [16384, 4096] x W [151936, 4096]: sampled dhidden rows through the
    oracle, and on every vocabulary row the identity sum_v dW[v] = 0 (each
    token's gradient sums to zero over the vocabulary)."""
    from vocab_wide_token_gb300 import inputs

    d = inputs.lmhead_workload(4, "cuda")
    h, W, y, w = d["hidden"], d["W"], d["labels"], d["weights"]
    err = cuda_lib.new_error_flag(h.device)
    lp, ent, rs = cuda_lib.lmhead_forward(h, W, y, IGN, dev_error=err)
    dh, dW = cuda_lib.lmhead_backward(h, W, y, w, rs, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.isfinite(dh).all() and torch.isfinite(dW).all()
    rng = np.random.default_rng(9)
    T = h.shape[0]
    rows = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 30, replace=False)]))
    z = olm.logits(to_oracle(h), to_oracle(W), rows)
    gref = oracle.backward(z, y[rows].cpu().numpy(), w[rows].double().cpu().numpy(), IGN)
    Wf = oracle.bf16_to_f64(to_oracle(W))
    rdh = gref @ Wf
    e1 = _frob_rel(dh[rows].double().cpu().numpy(), rdh)
    assert e1 <= 1e-3, e1
    # sum_v g[t, v] = 0 exactly; the fp16 gradient operand (2^15 q, one
    # rounding of 2^-12 relative per element, sum_v |q| <= 2) leaves at most
    # 2^-11 per token, times |w_t hidden_t| in the fp16 h', hence the bound
    # below (plus fp32 accumulation slack).
    colsum = dW.double().sum(dim=0)
    bound = 2.0**-10 * (w.double().abs()[:, None] * h.double().abs()).sum(dim=0)
    scale = dW.double().abs().sum(dim=0)
    assert torch.all(colsum.abs() <= bound + 1e-4 * scale + 1e-6)


def test_lmhead_backward_flags_fp16_range(cuda_lib):
    """The backward's 16-bit operands are fp16: a W entry or a weighted hidden
    value w_t hidden_t beyond 65504 cannot be represented and sets
    PSTAT_DEV_RANGE (values inside the range leave the flag clear)."""
    T, V, d = 130, 3000, 128
    h, W, y = _draw(T, V, d, 0.1, 31)
    w = torch.ones(T, device="cuda")
    lp, ent, rs = cuda_lib.lmhead_forward(h, W, y, IGN)
    err = cuda_lib.new_error_flag(h.device)
    cuda_lib.lmhead_backward(h, W, y, w, rs, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    w2 = w.clone()
    w2[7] = 1e5 / float(h[7].float().abs().max())  # |w h| reaches 1e5 on row 7
    err = cuda_lib.new_error_flag(h.device)
    cuda_lib.lmhead_backward(h, W, y, w2, rs, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() & cuda_lib.DEV_RANGE
    W2 = W.clone()
    W2[11, 5] = 1e5
    err = cuda_lib.new_error_flag(h.device)
    cuda_lib.lmhead_backward(h, W2, y, w, rs, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() & cuda_lib.DEV_RANGE
