"""Batch invariance, bit for bit: a row's logprob, entropy and dlogits are the
same bits whether it is computed alone, inside a batch of 7 or 512, or in the
full batch of 8192, at any position (the batch-invariance definition of the
torchtitan batch-invariant GDN README: a token's logprob must not depend on
the batch it sits in).  GPU against GPU; no oracle needed."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
IGN = -100


def _bits(x):
    return x.contiguous().view(torch.int16 if x.element_size() == 2 else torch.int32)


def _eval(pstat, z, y, w, bounds=None):
    lp, ent, rs = pstat.forward(z, y, IGN, bounds)
    g = pstat.backward(z, y, w, rs, IGN)
    return lp, ent, g


@pytest.fixture(scope="module")
def data():
    from vocab_wide_token_gb300 import inputs
    return inputs.fwdbwd_workload(2, "cuda")


@pytest.mark.parametrize("bounds", [None, [0, 50000, 100000, 151936]])
def test_rows_bitwise_across_batches(cuda_lib, data, bounds):
    z, y, w = data["logits"], data["labels"], data["weights"]
    T = z.shape[0]
    lp, ent, g = _eval(cuda_lib, z, y, w, bounds)
    rng = np.random.default_rng(7)
    probes = [0, 3, 4095, 8191] + rng.choice(T, 16, replace=False).tolist()
    for p in probes:
        ref = (_bits(lp[p:p + 1]), _bits(ent[p:p + 1]), _bits(g[p]))
        cases = []
        cases.append((slice(p, p + 1), 0))                     # alone
        for B in (7, 512):
            start = max(0, min(p - (p * 31 % B), T - B))       # contiguous slice, varied position
            cases.append((slice(start, start + B), p - start))
        for B in (7, 512):                                     # gathered copy, probe at varied slot
            others = torch.from_numpy(rng.choice(T, B - 1, replace=False)).to(z.device)
            slot = int(rng.integers(0, B))
            idx = torch.cat([others[:slot], torch.tensor([p], device=z.device), others[slot:]])
            cases.append((idx, slot))
        for sel, pos in cases:
            zz, yy, ww = z[sel], y[sel], w[sel]
            if not isinstance(sel, slice):
                zz = zz.contiguous()
            l2, e2, g2 = _eval(cuda_lib, zz, yy, ww, bounds)
            assert torch.equal(_bits(l2[pos:pos + 1]), ref[0]), (p, sel, "logprob")
            assert torch.equal(_bits(e2[pos:pos + 1]), ref[1]), (p, sel, "entropy")
            assert torch.equal(_bits(g2[pos]), ref[2]), (p, sel, "dlogits")


def test_repeat_calls_bitwise(cuda_lib, data):
    z, y, w = data["logits"][:2048], data["labels"][:2048], data["weights"][:2048]
    a = _eval(cuda_lib, z, y, w)
    b = _eval(cuda_lib, z, y, w)
    for x1, x2 in zip(a, b):
        assert torch.equal(_bits(x1), _bits(x2))
