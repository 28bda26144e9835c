"""Loss-side epilogue against the float64 oracle (oracle/policy.py): the
trainer/rollout mismatch metrics and the clipped-ratio surrogate, including a
full policy-gradient step (forward, surrogate weights, backward) checked
against the oracle's chain rule."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import policy as opol
from helpers import assert_grad_close, to_oracle

pytestmark = pytest.mark.gpu
IGN = -100


@pytest.mark.parametrize("T", [1, 7, 1000, 100003])
def test_diff_metrics(cuda_lib, T):
    g = torch.Generator(device="cuda").manual_seed(T)
    pi = -5 * torch.rand(T, generator=g, device="cuda")
    mu = pi.clone()
    flip = torch.rand(T, generator=g, device="cuda") < 0.3
    mu[flip] += 1e-3 * torch.randn(int(flip.sum()), generator=g, device="cuda")
    y = torch.randint(0, 10, (T,), generator=g, device="cuda")
    y[torch.rand(T, generator=g, device="cuda") < 0.1] = IGN
    out = cuda_lib.logprob_diff_metrics(pi, mu, y, IGN).cpu().numpy()
    ref = opol.diff_metrics(pi.cpu().numpy(), mu.cpu().numpy(), y.cpu().numpy(), IGN)
    for i, k in enumerate(["mean", "abs_mean", "max", "different"]):
        r = ref[k]
        if math.isnan(r):
            assert math.isnan(out[i])
        else:
            assert abs(out[i] - r) <= 1e-6 * max(abs(r), 1e-30) + 1e-12, (k, out[i], r)
    again = cuda_lib.logprob_diff_metrics(pi, mu, y, IGN)
    assert torch.equal(again.view(torch.int32), torch.from_numpy(out).to("cuda").view(torch.int32))


def test_diff_metrics_degenerate(cuda_lib):
    z = torch.zeros(3, device="cuda")
    out = cuda_lib.logprob_diff_metrics(z, -z, None).cpu().numpy()   # +0 vs -0
    assert out[0] == 0 and out[1] == 0 and out[2] == 0 and out[3] == 1.0
    y = torch.full((3,), IGN, device="cuda")
    out = cuda_lib.logprob_diff_metrics(z, z, y, IGN).cpu().numpy()
    assert math.isnan(out[0]) and out[2] == 0 and math.isnan(out[3])


@pytest.mark.parametrize("T", [5, 4097])
def test_clipped_surrogate(cuda_lib, T):
    g = torch.Generator(device="cuda").manual_seed(T + 1)
    old = -2 + torch.randn(T, generator=g, device="cuda")
    pi = old + 0.4 * torch.randn(T, generator=g, device="cuda")
    adv = torch.randn(T, generator=g, device="cuda")
    y = torch.randint(0, 5, (T,), generator=g, device="cuda")
    y[0] = IGN
    loss, w = cuda_lib.clipped_surrogate(pi, old, adv, y, 0.2, 0.28, 0.5, IGN)
    rl, rw = opol.clipped_surrogate(pi.cpu().numpy(), old.cpu().numpy(), adv.cpu().numpy(),
                                    y.cpu().numpy(), 0.2, 0.28, 0.5, IGN)
    l, ww = loss.double().cpu().numpy(), w.double().cpu().numpy()
    r = np.exp(pi.double().cpu().numpy() - old.double().cpu().numpy())
    # where the branch (clipped or not) is decided by a margin, both must agree;
    # within 1e-5 of a kink either branch's value is a correct result
    a = adv.double().cpu().numpy()
    rc = np.clip(r, 0.8, 1.28)
    margin = np.abs(r * a - rc * a) > 1e-5 * np.abs(a)
    assert np.allclose(l[margin], rl[margin], rtol=1e-5, atol=1e-7)
    assert np.allclose(ww[margin], rw[margin], rtol=1e-5, atol=1e-7)
    for t in np.flatnonzero(~margin):
        assert np.isclose(ww[t], -0.5 * a[t] * r[t], rtol=1e-5) or ww[t] == 0.0
    assert l[0] == 0 and ww[0] == 0


def test_policy_gradient_step(cuda_lib):
    """forward -> surrogate weights -> backward equals the oracle chain rule
    d loss / d z_t = (d loss_t / d logprob_t)(onehot - softmax)."""
    from vocab_wide_token_gb300 import inputs

    d = inputs.fwdbwd_workload(2, "cuda", T=64, V=20000)
    z, y = d["logits"], d["labels"]
    g = torch.Generator(device="cuda").manual_seed(3)
    lp, ent, rs = cuda_lib.forward(z, y, IGN)
    old = lp + 0.3 * torch.randn(64, generator=g, device="cuda")
    adv = torch.randn(64, generator=g, device="cuda")
    loss, w = cuda_lib.clipped_surrogate(lp, old, adv, y)
    gl = cuda_lib.backward(z, y, w, rs, IGN)
    torch.cuda.synchronize()
    ref = oracle.forward(to_oracle(z), y.cpu().numpy(), IGN)
    _, rw = opol.clipped_surrogate(ref["logprob"], old.double().cpu().numpy(),
                                   adv.double().cpu().numpy(), y.cpu().numpy())
    # the branch decision compares GPU and oracle logprobs that differ by ~1e-6:
    # keep rows whose decision has margin
    r = np.exp(ref["logprob"] - old.double().cpu().numpy())
    a = adv.double().cpu().numpy()
    keep = np.abs(r * a - np.clip(r, 0.8, 1.28) * a) > 1e-4 * np.abs(a) + 1e-12
    gref = oracle.backward(to_oracle(z[keep]), y[keep].cpu().numpy(), rw[keep], IGN)
    assert_grad_close(gl[torch.from_numpy(keep).cuda()], gref, torch.bfloat16, "policy step")
