"""Full log-softmax output (pstat_log_softmax) against the float64 oracle,
including masked columns, ragged sizes, unaligned rows, bf16 rounding and
bitwise batch invariance."""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import TOL_FWD, bf16_round, bf16_ulp, to_oracle

pytestmark = pytest.mark.gpu


def _close(out, ref, in_dtype, out_dtype):
    a = out.double().cpu().numpy()
    fin = np.isfinite(ref)
    assert np.all(np.isneginf(a[~fin]) | np.isnan(a[~fin]))
    if out_dtype == torch.float32:
        tol = TOL_FWD[in_dtype] + 2 * np.spacing(np.abs(ref[fin]).astype(np.float32)).astype(np.float64)
        assert np.all(np.abs(a[fin] - ref[fin]) <= tol), float(np.max(np.abs(a[fin] - ref[fin]) - tol))
    else:
        br = bf16_round(ref[fin])
        assert np.all(np.abs(a[fin] - br) <= bf16_ulp(ref[fin]))


@pytest.mark.parametrize("in_dtype,out_dtype", [(torch.float32, torch.float32),
                                                (torch.bfloat16, torch.bfloat16),
                                                (torch.bfloat16, torch.float32),
                                                (torch.float32, torch.bfloat16)])
@pytest.mark.parametrize("V", [7, 1001, 10007])
def test_log_softmax(cuda_lib, in_dtype, out_dtype, V):
    g = torch.Generator(device="cuda").manual_seed(V)
    T = 33
    z = (3 * torch.randn(T, V, generator=g, device="cuda")).float()
    if V > 10:
        z[4, ::3] = -math.inf
    z = z.to(in_dtype)
    out = cuda_lib.log_softmax(z, None, None, out_dtype)
    torch.cuda.synchronize()
    _close(out, oracle.log_softmax(to_oracle(z)), in_dtype, out_dtype)


def test_log_softmax_from_rowstats_unaligned_and_invariant(cuda_lib):
    g = torch.Generator(device="cuda").manual_seed(5)
    T, V = 50, 151936
    big = (2 * torch.randn(T, V + 3, generator=g, device="cuda")).to(torch.bfloat16)
    z = big[:, 1:1 + V]                       # rows off 16-byte boundaries
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    lp, ent, rs = cuda_lib.forward(z, y)
    out = cuda_lib.log_softmax(z, rs)
    out2 = cuda_lib.log_softmax(z.contiguous())
    one = cuda_lib.log_softmax(z[7:8].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.equal(one[0].view(torch.int16), out[7].view(torch.int16))
    rows = [0, 7, 49]
    _close(out[rows], oracle.log_softmax(to_oracle(z[rows])), torch.bfloat16, torch.bfloat16)
    # log p at the label is the logprob
    assert torch.allclose(out.float()[torch.arange(T), y], lp, atol=0.05)


def test_log_softmax_empty_row_flags(cuda_lib):
    z = torch.randn(3, 100, device="cuda")
    z[1] = -math.inf
    err = cuda_lib.new_error_flag(z.device)
    out = cuda_lib.log_softmax(z, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() & cuda_lib.DEV_EMPTY_ROW
    assert torch.all(torch.isnan(out[1])) and torch.all(torch.isfinite(out[0]))
