"""Parity of the CUDA path (through the C ABI) with the float64 oracle on
small and medium inputs that span several chunks and a ragged tail, plus the
edge cases the method has.  Tolerances: tests/helpers.py."""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_forward_close, assert_grad_close, to_oracle

pytestmark = pytest.mark.gpu
IGN = -100


def _run(pstat, z, y, w=None, bounds=None, out_dtype=None):
    err = pstat.new_error_flag(z.device)
    lp, ent, rs = pstat.forward(z, y, IGN, bounds, dev_error=err)
    g = pstat.backward(z, y, w, rs, IGN, out_dtype=out_dtype, dev_error=err) if w is not None else None
    torch.cuda.synchronize()
    return lp, ent, rs, g, int(err.item())


def _check(pstat, z, y, w, bounds=None, out_dtype=None, what=""):
    lp, ent, rs, g, err = _run(pstat, z, y, w, bounds, out_dtype)
    zo = to_oracle(z)
    yo = y.cpu().numpy()
    ref = oracle.forward(zo, yo, IGN)
    assert_forward_close(lp, ent, ref, z.dtype, what=what)
    # row statistics: ln S + M is the log-partition
    L = (rs[:, 0].double() + rs[:, 1].double()).cpu().numpy()
    Lref = ref["M"] + ref["logS"]
    fin = np.isfinite(Lref)
    assert np.allclose(L[fin], Lref[fin], rtol=0, atol=10 * (1e-5 if z.dtype == torch.float32 else 1e-4))
    if w is not None:
        gref = oracle.backward(zo, yo, w.double().cpu().numpy(), IGN)
        assert_grad_close(g, gref, out_dtype or z.dtype, what=what)
    return err


def test_tiny_config(cuda_lib):
    """64 x 1000 fp32, N(0, 3^2), 5 ignored labels, shards 512/488, weights N(0, 1)."""
    from vocab_wide_token_gb300 import inputs

    d = inputs.tiny(0, "cuda")
    err = _check(cuda_lib, d["logits"], d["labels"], d["weights"], d["shard_bounds"],
                 torch.float32, "tiny")
    assert err == 0
    # the single-shard path agrees too
    assert _check(cuda_lib, d["logits"], d["labels"], d["weights"], None, torch.float32) == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("V,bounds", [
    (10007, None),                      # several chunks, ragged tail
    (10007, [0, 4096, 10007]),
    (10007, [0, 513, 6000, 10007]),     # shard starts not 16-byte aligned
    (1001, None), (8, None), (7, None), (1, None),
    (151936, [0, 50000, 100000, 151936]),
])
def test_multi_chunk_ragged(cuda_lib, dtype, V, bounds):
    g = torch.Generator(device="cuda").manual_seed(V)
    T = 37
    z = (2.5 * torch.randn(T, V, generator=g, device="cuda")).to(dtype)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    y[3] = IGN
    w = torch.randn(T, generator=g, device="cuda")
    w[5] = 0.0
    out = torch.float32 if dtype == torch.float32 else torch.bfloat16
    assert _check(cuda_lib, z, y, w, bounds, out, f"V={V} {dtype}") == 0
    if dtype == torch.float32:
        assert _check(cuda_lib, z, y, w, bounds, torch.bfloat16, f"V={V} f32->bf16") == 0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("offset", [1, 3, 8])
def test_unaligned_rows(cuda_lib, dtype, offset):
    """Rows that start off a 16-byte boundary (a column slice of a wider
    tensor, odd row stride) take the element-load path with the same result."""
    g = torch.Generator(device="cuda").manual_seed(offset)
    T, V = 19, 9001
    big = (2.0 * torch.randn(T, V + offset + 5, generator=g, device="cuda")).to(dtype)
    z = big[:, offset:offset + V]
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    w = torch.randn(T, generator=g, device="cuda")
    assert _check(cuda_lib, z, y, w, [0, 4001, V], None, f"offset {offset}") == 0
    # bitwise equal to the same rows stored contiguously (numerics do not see alignment)
    lp1, ent1, _, g1, _ = _run(cuda_lib, z, y, w, [0, 4001, V])
    lp2, ent2, _, g2, _ = _run(cuda_lib, z.contiguous(), y, w, [0, 4001, V])
    assert torch.equal(lp1.view(torch.int32), lp2.view(torch.int32))
    assert torch.equal(ent1.view(torch.int32), ent2.view(torch.int32))
    assert torch.equal(g1.contiguous().view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       g2.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_masked_and_degenerate_rows(cuda_lib, dtype):
    T, V = 12, 20000
    g = torch.Generator(device="cuda").manual_seed(11)
    z = (2.0 * torch.randn(T, V, generator=g, device="cuda")).float()
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    z[0, :] = 0.0                          # uniform row
    z[1, :] = -math.inf
    z[1, 123] = 1.5                        # single finite entry, label on it
    y[1] = 123
    z[2, :4096 if dtype == torch.bfloat16 else 2048] = -math.inf  # a whole chunk masked
    z[3, ::3] = -math.inf                  # partially masked row
    y[3] = 1
    z[4, 7] = -math.inf                    # label on a -inf column: logprob -inf
    y[4] = 7
    z[5, :10000] = -math.inf               # whole first shard masked
    y[5] = 10001
    y[6] = IGN
    z[7] = z[7] + 30.0                     # shifted row
    z = z.to(dtype)
    w = torch.randn(T, generator=g, device="cuda")
    out = torch.float32 if dtype == torch.float32 else torch.bfloat16
    err = _check(cuda_lib, z, y, w, [0, 10000, V], out, "degenerate")
    assert err == 0
    lp, ent, _, gg, _ = _run(cuda_lib, z, y, w, [0, 10000, V], out)
    assert abs(lp[0].item() + math.log(V)) < 1e-4 and abs(ent[0].item() - math.log(V)) < 1e-4
    assert lp[1].item() == 0.0 and ent[1].item() == 0.0
    assert lp[4].item() == -math.inf
    assert lp[6].item() == 0.0 and torch.all(gg[6] == 0)


def test_huge_fp32_logits(cuda_lib):
    """|z| up to 1e4 in fp32: the chunk shift keeps every exponent exact."""
    g = torch.Generator(device="cuda").manual_seed(21)
    T, V = 9, 5000
    z = torch.randn(T, V, generator=g, device="cuda") * 3.0
    z[:3] += 1e4
    z[3:6] -= 1e4
    z[6, 17] = 1e4
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    w = torch.randn(T, generator=g, device="cuda")
    assert _check(cuda_lib, z, y, w, [0, 2500, V], torch.float32, "huge") == 0


def test_device_errors_are_flagged_not_trapped(cuda_lib):
    T, V = 4, 3000
    z = torch.randn(T, V, device="cuda")
    z[2] = -math.inf                       # empty row
    y = torch.tensor([5, V, 3, -7], device="cuda")   # V and -7 are bad labels
    w = torch.ones(T, device="cuda")
    lp, ent, rs, g, err = _run(cuda_lib, z, y, w)
    assert err & cuda_lib.DEV_BAD_LABEL and err & cuda_lib.DEV_EMPTY_ROW
    assert not math.isnan(lp[0].item())
    assert math.isnan(lp[1].item()) and math.isnan(lp[2].item()) and math.isnan(lp[3].item())
    assert torch.all(torch.isnan(g[1])) and torch.all(torch.isnan(g[2]))
    assert not torch.any(torch.isnan(g[0]))


def test_all_rows_ignored_and_empty_batch(cuda_lib):
    z = torch.randn(5, 777, device="cuda").to(torch.bfloat16)
    y = torch.full((5,), IGN, device="cuda")
    w = torch.randn(5, device="cuda")
    lp, ent, rs, g, err = _run(cuda_lib, z, y, w)
    assert err == 0 and torch.all(lp == 0) and torch.all(g == 0)
    assert not torch.any(torch.signbit(g.float()))
    ref = oracle.forward(to_oracle(z), y.cpu().numpy(), IGN)
    assert np.allclose(ent.double().cpu().numpy(), ref["entropy"], atol=1e-4)
    z0 = torch.empty(0, 777, device="cuda")
    lp, ent, rs = cuda_lib.forward(z0, torch.empty(0, dtype=torch.int64, device="cuda"))
    assert lp.numel() == 0


def test_backward_recomputes_rowstats(cuda_lib):
    """rowstats=NULL recomputes (M, ln S) through the forward kernels: same bits."""
    g = torch.Generator(device="cuda").manual_seed(31)
    z = (2.0 * torch.randn(33, 12345, generator=g, device="cuda")).to(torch.bfloat16)
    y = torch.randint(0, 12345, (33,), generator=g, device="cuda")
    w = torch.randn(33, generator=g, device="cuda")
    _, _, rs = cuda_lib.forward(z, y)
    g1 = cuda_lib.backward(z, y, w, rs)
    g2 = cuda_lib.backward(z, y, w, None)
    assert torch.equal(g1.view(torch.int16), g2.view(torch.int16))


def test_autograd_function(cuda_lib):
    g = torch.Generator(device="cuda").manual_seed(41)
    z = (2.0 * torch.randn(16, 3000, generator=g, device="cuda")).requires_grad_(True)
    y = torch.randint(0, 3000, (16,), generator=g, device="cuda")
    y[2] = IGN
    lp, ent = cuda_lib.policy_stats(z, y)
    adv = torch.randn(16, generator=g, device="cuda")
    (lp * adv).sum().backward()
    ref = oracle.backward(to_oracle(z.detach()), y.cpu().numpy(), adv.double().cpu().numpy(), IGN)
    assert_grad_close(z.grad, ref, torch.float32, "autograd")
    assert not ent.requires_grad


def test_forward_past_256_chunks(cuda_lib):
    # More than 256 chunks per row: pstat_forward takes the chunk-statistics
    # kernel and the combine (the one-kernel path holds 256 records per row),
    # the backward's recompute does the same, and the single pass refuses.
    V = 256 * 4096 + 1000
    T = 6
    g = torch.Generator(device="cuda").manual_seed(257)
    z = (2.0 * torch.randn(T, V, generator=g, device="cuda")).to(torch.bfloat16)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    y[2] = IGN
    w = torch.randn(T, generator=g, device="cuda")
    lp, ent, rs = cuda_lib.forward(z, y, IGN)
    g1 = cuda_lib.backward(z, y, w, rs, IGN)
    g2 = cuda_lib.backward(z, y, w, None, IGN)
    torch.cuda.synchronize()
    assert torch.equal(g1.view(torch.int16), g2.view(torch.int16))
    ref = oracle.forward(to_oracle(z), y.cpu().numpy(), IGN)
    assert_forward_close(lp, ent, ref, torch.bfloat16, what="V > 256 chunks")
    with pytest.raises(cuda_lib.PstatError):
        cuda_lib.forward_backward(z, y, w, IGN)


def test_bad_output_tensors_raise_before_launch(cuda_lib):
    """Outputs on the host, of the wrong size or type, and inputs on the host
    are rejected by the binding; nothing is launched and the device stays
    usable."""
    T, V = 16, 1000
    z = torch.randn(T, V, device="cuda").to(torch.bfloat16)
    y = torch.randint(0, V, (T,), device="cuda")
    w = torch.randn(T, device="cuda")
    lp, ent, rs = cuda_lib.forward(z, y, IGN)
    host = (torch.empty(T), torch.empty(T), torch.empty(T, 2))
    with pytest.raises(ValueError):
        cuda_lib.forward(z, y, IGN, out=host)
    with pytest.raises(ValueError):
        cuda_lib.forward_backward(z, y, w, IGN, dlogits=torch.empty(T, V - 1, device="cuda",
                                                                   dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        cuda_lib.backward(z, y, w.cpu(), rs, IGN)
    with pytest.raises(ValueError):
        cuda_lib.backward(z, y, w, rs[:, :1], IGN)
    with pytest.raises(ValueError):
        cuda_lib.log_softmax(z, rs, out=torch.empty(T, V, device="cuda", dtype=torch.float16))
    with pytest.raises(ValueError):
        cuda_lib.forward(z, y, IGN, dev_error=torch.zeros(1, dtype=torch.int64, device="cuda"))
    h = torch.randn(T, 64, device="cuda").to(torch.bfloat16)
    W = torch.randn(V, 64, device="cuda").to(torch.bfloat16)
    lph, enth, rsh = cuda_lib.lmhead_forward(h, W, y, IGN)
    with pytest.raises(ValueError):
        cuda_lib.lmhead_backward(h, W, y, w, rsh, IGN, dW=torch.zeros(V - 1, 64, device="cuda"))
    # the device is still fine
    lp2, ent2, rs2 = cuda_lib.forward(z, y, IGN)
    torch.cuda.synchronize()
    assert torch.equal(lp, lp2) and torch.equal(ent, ent2)


def test_bounded_wait_times_out_and_the_context_stays_usable(cuda_lib):
    """A kernel's wait on an mbarrier that nothing arrives at gives up after
    its limit and reports PSTAT_DEV_TIMEOUT instead of hanging; no copy is in
    flight, and the next calls run normally."""
    import time

    t0 = time.perf_counter()
    bits = cuda_lib.selftest_wait_timeout("cuda", 20_000_000)  # 20 ms
    dt = time.perf_counter() - t0
    assert bits == cuda_lib.DEV_TIMEOUT
    assert dt < 5.0
    z = torch.randn(8, 3000, device="cuda")
    y = torch.randint(0, 3000, (8,), device="cuda")
    err = cuda_lib.new_error_flag(z.device)
    lp, ent, rs = cuda_lib.forward(z, y, -100, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    ref = oracle.forward(z.cpu().numpy(), y.cpu().numpy(), -100)
    assert_forward_close(lp, ent, ref, torch.float32, what="after the timeout self-test")
