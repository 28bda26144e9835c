"""pstat_forward_backward (one pass over the logits) against the two-call
path pstat_forward + pstat_backward -- bit for bit -- and against the float64
oracle directly, on the edge cases and at full size."""
import math

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_forward_close, assert_grad_close, to_oracle

pytestmark = pytest.mark.gpu
IGN = -100


def _bits(x):
    x = x.contiguous()
    return x.view(torch.int16 if x.element_size() == 2 else torch.int32)


def _same_as_two_calls(pstat, z, y, w, bounds=None, out_dtype=None):
    e1 = pstat.new_error_flag(z.device)
    e2 = pstat.new_error_flag(z.device)
    lp, ent, rs = pstat.forward(z, y, IGN, bounds, dev_error=e1)
    g = pstat.backward(z, y, w, rs, IGN, out_dtype=out_dtype, dev_error=e1)
    lp2, ent2, rs2, g2 = pstat.forward_backward(z, y, w, IGN, bounds, out_dtype, dev_error=e2)
    torch.cuda.synchronize()
    for a, b, name in ((lp, lp2, "logprob"), (ent, ent2, "entropy"), (rs, rs2, "rowstats"),
                       (g, g2, "dlogits")):
        assert torch.equal(_bits(a), _bits(b)), name
    assert e1.item() == e2.item()
    return lp2, ent2, rs2, g2, e2.item()


@pytest.mark.parametrize("dtype,out_dtype", [(torch.bfloat16, torch.bfloat16),
                                             (torch.float32, torch.float32),
                                             (torch.float32, torch.bfloat16)])
@pytest.mark.parametrize("V,bounds", [(10007, None), (10007, [0, 513, 6000, 10007]),
                                      (1001, None), (8, None), (7, None), (1, None),
                                      (30000, None), (70000, None), (106000, None),
                                      (151936, None),
                                      (151936, [0, 50000, 100000, 151936])])
def test_fused_bitwise_equals_two_calls(cuda_lib, dtype, out_dtype, V, bounds):
    # V = 106000 is 26 bf16 (52 fp32) chunks, 2 (4) per warp: the forward
    # folds with a warp of its own, as for 39 chunks over three shards.
    # With V = 151936 and one shard, each warp holds 2 or 3 chunks of a row.
    # Row 5's first third is -inf, so a warp whose first chunk of that row is
    # masked takes the clamped exponent pass first on its later, unmasked
    # chunks in the forward, and the unclamped one in the single pass.  The
    # two must agree bit for bit.
    g = torch.Generator(device="cuda").manual_seed(V + 17)
    T = 300
    z = (2.5 * torch.randn(T, V, generator=g, device="cuda")).float()
    if V > 20:
        z[5, : V // 3] = -math.inf          # masked first third
        z[6, ::5] = -math.inf
    z = z.to(dtype)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    y[3] = IGN
    if V > 20:
        y[6] = 1
    w = torch.randn(T, generator=g, device="cuda")
    w[4] = 0.0
    lp, ent, rs, gg, err = _same_as_two_calls(cuda_lib, z, y, w, bounds, out_dtype)
    assert err == 0
    zo, yo = to_oracle(z), y.cpu().numpy()
    ref = oracle.forward(zo, yo, IGN)
    assert_forward_close(lp, ent, ref, dtype, what=f"fused V={V}")
    gref = oracle.backward(zo, yo, w.double().cpu().numpy(), IGN)
    assert_grad_close(gg, gref, out_dtype, f"fused V={V}")


# A NaN payload no kernel produces: a store outside the T x V block of a
# wider output buffer would overwrite it.
CANARY16 = 0x7FA5
CANARY32 = 0x7FC0A5A5


def _canary_buffer(T, width, dtype):
    if dtype == torch.bfloat16:
        return torch.full((T, width), CANARY16, dtype=torch.int16, device="cuda").view(dtype)
    return torch.full((T, width), CANARY32, dtype=torch.int32, device="cuda").view(dtype)


def _assert_canary_intact(buf, c0, c1, what):
    """Columns outside [c0, c1) of every row still hold the canary."""
    bits = _bits(buf)
    want = CANARY16 if buf.element_size() == 2 else CANARY32
    outside = torch.cat([bits[:, :c0], bits[:, c1:]], dim=1)
    bad = outside != want
    assert not bool(bad.any()), f"{what}: {int(bad.sum())} elements outside the output overwritten"


@pytest.mark.parametrize("offset", [1, 3])
def test_fused_unaligned_rows_and_outputs(cuda_lib, offset):
    g = torch.Generator(device="cuda").manual_seed(offset)
    T, V = 40, 9001
    big = (2.0 * torch.randn(T, V + offset + 5, generator=g, device="cuda")).to(torch.bfloat16)
    z = big[:, offset:offset + V]
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    w = torch.randn(T, generator=g, device="cuda")
    lp, ent, rs = cuda_lib.forward(z, y, IGN)
    g1 = cuda_lib.backward(z, y, w, rs, IGN)
    outbig = _canary_buffer(T, V + 3, torch.bfloat16)
    dl = outbig[:, 1:1 + V]
    lp2, ent2, rs2, g2 = cuda_lib.forward_backward(z, y, w, IGN, dlogits=dl)
    torch.cuda.synchronize()
    assert torch.equal(_bits(lp), _bits(lp2)) and torch.equal(_bits(ent), _bits(ent2))
    assert torch.equal(_bits(g1), _bits(g2))
    _assert_canary_intact(outbig, 1, 1 + V, "forward_backward")


@pytest.mark.parametrize("dtype,out_dtype,V,lead,tail",
                         [(torch.bfloat16, torch.bfloat16, 9001, 1, 2),
                          (torch.bfloat16, torch.bfloat16, 151936, 8, 8),
                          (torch.float32, torch.float32, 10007, 3, 1),
                          (torch.float32, torch.bfloat16, 4096, 1, 7)])
def test_wider_outputs_keep_their_margins(cuda_lib, dtype, out_dtype, V, lead, tail):
    """pstat_backward, pstat_forward_backward and pstat_log_softmax writing
    into a view of a wider buffer (ld_out > V, first column at an offset)
    touch nothing outside their T x V block, and give the same bits as with
    a dense output."""
    T = 37
    g = torch.Generator(device="cuda").manual_seed(V + lead)
    z = (2.0 * torch.randn(T, V, generator=g, device="cuda")).to(dtype)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    y[2] = IGN
    w = torch.randn(T, generator=g, device="cuda")
    w[3] = 0.0
    lp, ent, rs = cuda_lib.forward(z, y, IGN)
    dense_b = cuda_lib.backward(z, y, w, rs, IGN, out_dtype=out_dtype)
    dense_l = cuda_lib.log_softmax(z, rs, out_dtype=out_dtype)
    width = lead + V + tail
    for name in ("backward", "forward_backward", "log_softmax"):
        buf = _canary_buffer(T, width, out_dtype)
        view = buf[:, lead:lead + V]
        if name == "backward":
            cuda_lib.backward(z, y, w, rs, IGN, out_dtype=out_dtype, out=view)
            dense = dense_b
        elif name == "forward_backward":
            cuda_lib.forward_backward(z, y, w, IGN, out_dtype=out_dtype, dlogits=view)
            dense = dense_b
        else:
            cuda_lib.log_softmax(z, rs, out_dtype=out_dtype, out=view)
            dense = dense_l
        torch.cuda.synchronize()
        _assert_canary_intact(buf, lead, lead + V, name)
        assert torch.equal(_bits(view), _bits(dense)), name


@pytest.mark.parametrize("dtype,V,offset,extra", [(torch.bfloat16, 1001, 0, 0),
                                                (torch.bfloat16, 1001, 1, 0),
                                                (torch.bfloat16, 4096, 1, 2),
                                                (torch.bfloat16, 151936, 0, 1),
                                                (torch.float32, 1001, 1, 0)])
def test_label_logit_at_row_edges(cuda_lib, dtype, V, offset, extra):
    """Labels on the first two and last two columns of rows whose starts fall
    on either half of a 4-byte word (odd row strides and view offsets): the
    label's logit is fetched as the aligned word that holds it, and where that
    word would reach outside the row it is loaded on its own."""
    T = 64
    g = torch.Generator(device="cuda").manual_seed(V + offset + extra)
    big = (2.0 * torch.randn(T, V + offset + extra, generator=g, device="cuda")).to(dtype)
    z = big[:, offset:offset + V]
    y = torch.empty(T, dtype=torch.int64, device="cuda")
    y[0::4], y[1::4], y[2::4], y[3::4] = 0, V - 1, 1, V - 2
    w = torch.randn(T, generator=g, device="cuda")
    err = cuda_lib.new_error_flag(z.device)
    lp, ent, rs = cuda_lib.forward(z, y, IGN, dev_error=err)
    lp2, ent2, rs2, g2 = cuda_lib.forward_backward(z, y, w, IGN, dev_error=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(_bits(lp), _bits(lp2)) and torch.equal(_bits(ent), _bits(ent2))
    zo, yo = to_oracle(z.contiguous()), y.cpu().numpy()
    ref = oracle.forward(zo, yo, IGN)
    assert_forward_close(lp2, ent2, ref, dtype, what=f"edge labels V={V}")
    gref = oracle.backward(zo, yo, w.double().cpu().numpy(), IGN)
    assert_grad_close(g2, gref, dtype, f"edge labels V={V}")


def test_fused_device_errors(cuda_lib):
    T, V = 4, 3000
    z = torch.randn(T, V, device="cuda")
    z[2] = -math.inf
    y = torch.tensor([5, V, 3, -7], device="cuda")
    w = torch.ones(T, device="cuda")
    lp, ent, rs, g, err = _same_as_two_calls(cuda_lib, z, y, w)
    assert err & cuda_lib.DEV_BAD_LABEL and err & cuda_lib.DEV_EMPTY_ROW
    assert torch.all(torch.isnan(g[1])) and torch.all(torch.isnan(g[2]))


def test_fused_rows_beyond_the_label_cache(cuda_lib):
    # Each CTA keeps the labels and weights of its first 384 rows in shared
    # memory and reads later rows' labels from global memory: give every CTA
    # more rows than that, with ignored, zero-weight and bad labels among the
    # late rows, and check the whole batch bit for bit against the two calls.
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T, V = sms * 390 + 7, 1500
    g = torch.Generator(device="cuda").manual_seed(11)
    z = (2.0 * torch.randn(T, V, generator=g, device="cuda")).to(torch.bfloat16)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    w = torch.randn(T, generator=g, device="cuda")
    late = torch.arange(sms * 384, T, device="cuda")
    y[late[::97]] = IGN
    w[late[5::89]] = 0.0
    y[late[-3]] = V + 2
    lp, ent, rs, gg, err = _same_as_two_calls(cuda_lib, z, y, w)
    assert err & cuda_lib.DEV_BAD_LABEL
    rows = late[[0, 1, 50, 400, -1]].cpu()
    zo = to_oracle(z[rows])
    yo = y[rows].cpu().numpy()
    ref = oracle.forward(zo, yo, IGN)
    assert_forward_close(lp[rows.cuda()], ent[rows.cuda()], ref, torch.bfloat16,
                         what="rows past the label cache")
    assert_grad_close(gg[rows.cuda()], oracle.backward(zo, yo, w[rows].double().cpu().numpy(), IGN),
                      torch.bfloat16, "rows past the label cache")


@pytest.mark.parametrize("dtype,V", [(torch.bfloat16, 300000), (torch.bfloat16, 700000),
                                     (torch.float32, 150000), (torch.float32, 350000)])
def test_fused_long_rows(cuda_lib, dtype, V):
    # 74 and 171 chunks per row (up to 6 and 14 per warp of a CTA), a masked half row
    # and an ignored label: bit for bit against the two calls, and the oracle
    # on sampled rows.
    g = torch.Generator(device="cuda").manual_seed(V)
    T = 40
    z = (2.0 * torch.randn(T, V, generator=g, device="cuda")).to(dtype)
    z[3, V // 2:] = -math.inf
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    y[1] = IGN
    w = torch.randn(T, generator=g, device="cuda")
    lp, ent, rs, gg, err = _same_as_two_calls(cuda_lib, z, y, w)
    assert err == 0
    rows = np.array([0, 3, 39])
    zo, yo = to_oracle(z[rows]), y[rows].cpu().numpy()
    assert_forward_close(lp[rows], ent[rows], oracle.forward(zo, yo, IGN), dtype,
                         what=f"long rows V={V}")
    assert_grad_close(gg[rows], oracle.backward(zo, yo, w[rows].double().cpu().numpy(), IGN),
                      dtype, f"long rows V={V}")


def test_fused_tiny_config_against_oracle(cuda_lib):
    from vocab_wide_token_gb300 import inputs

    d = inputs.tiny(0, "cuda")
    z, y, w, b = d["logits"], d["labels"], d["weights"], d["shard_bounds"]
    lp, ent, rs, g = cuda_lib.forward_backward(z, y, w, IGN, b, torch.float32)
    torch.cuda.synchronize()
    zo, yo = z.cpu().numpy(), y.cpu().numpy()
    assert_forward_close(lp, ent, oracle.forward(zo, yo, IGN), torch.float32, what="tiny")
    assert_grad_close(g, oracle.backward(zo, yo, w.double().cpu().numpy(), IGN), torch.float32,
                      "tiny")


def test_fused_full_size_and_batch_invariance(cuda_lib):
    """T=8192, V=151936 bf16 (the benchmark workload): bitwise equal to the
    two-call path on every row; sampled rows alone give the same bits."""
    from vocab_wide_token_gb300 import inputs

    d = inputs.fwdbwd_workload(2, "cuda")
    z, y, w = d["logits"], d["labels"], d["weights"]
    lp, ent, rs, g, err = _same_as_two_calls(cuda_lib, z, y, w)
    assert err == 0
    for p in (0, 4095, 8191):
        l1, e1, r1, g1 = cuda_lib.forward_backward(z[p:p + 1], y[p:p + 1], w[p:p + 1])
        torch.cuda.synchronize()
        assert torch.equal(_bits(l1), _bits(lp[p:p + 1]))
        assert torch.equal(_bits(g1[0]), _bits(g[p]))
    rows = np.array([0, 1, 77, 4095, 8191])
    zo, yo = to_oracle(z[rows]), y[rows].cpu().numpy()
    assert_forward_close(lp[rows], ent[rows], oracle.forward(zo, yo, IGN), torch.bfloat16)
    assert_grad_close(g[rows], oracle.backward(zo, yo, w[rows].double().cpu().numpy(), IGN),
                      torch.bfloat16, "full")


@pytest.mark.parametrize("T,block", [(1000, 300), (64, 1024), (1, 1)])
def test_from_host_equals_device_call(cuda_lib, T, block):
    # forward_backward_from_host stages row blocks through a double buffer on a
    # side stream; every output must equal the one-call result bit for bit.
    V = 4099
    g = torch.Generator().manual_seed(T)
    zh = (2.0 * torch.randn(T, V, generator=g)).to(torch.bfloat16).pin_memory()
    yh = torch.randint(0, V, (T,), generator=g).pin_memory()
    wh = torch.randn(T, generator=g).pin_memory()
    if T > 2:
        yh[1] = IGN
    ref = cuda_lib.forward_backward(zh.cuda(), yh.cuda(), wh.cuda(), IGN)
    got = cuda_lib.forward_backward_from_host(zh, yh, wh, IGN, block_rows=block)
    torch.cuda.synchronize()
    for a, b, name in zip(ref, got, ("logprob", "entropy", "rowstats", "dlogits")):
        assert torch.equal(_bits(a), _bits(b)), name
    # the same with dlogits also copied back to pinned host memory block by block
    gh = torch.full((T, V), float("nan"), dtype=torch.bfloat16).pin_memory()
    got2 = cuda_lib.forward_backward_from_host(zh, yh, wh, IGN, block_rows=block,
                                               dlogits_host=gh)
    torch.cuda.current_stream().synchronize()
    assert torch.equal(_bits(gh), _bits(ref[3].cpu()))
    assert torch.equal(_bits(got2[0]), _bits(ref[0]))
