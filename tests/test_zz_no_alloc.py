"""pstat_forward_noalloc: the forward statistics for callers that cannot
allocate device memory (allocation would synchronise the device, or their
host owns all device memory through its own pool, or they have no allocator).

It takes no workspace; its scratch is a fixed array inside libpstat.so.  The
test calls it through the C ABI (ctypes binding) twice in a row on different
inputs and checks each result against the workspace entry point pstat_forward
with the parity tolerances the other tests use (the kernels are the same, so
the results are in fact expected to be identical bit for bit), and checks that
a problem larger than the fixed scratch is refused before any launch.

This file is named so that pytest collects it last."""
import pytest
import torch

from helpers import TOL_FWD

pytestmark = pytest.mark.gpu
IGN = -100


def _draw(seed, T, V, dtype):
    g = torch.Generator(device="cuda").manual_seed(seed)
    z = (2.0 * torch.randn(T, V, generator=g, device="cuda")).to(dtype)
    y = torch.randint(0, V, (T,), generator=g, device="cuda")
    y[1] = IGN
    return z, y


def _same(a, b, tol):
    assert torch.allclose(a, b, rtol=0, atol=tol, equal_nan=True)


@pytest.mark.parametrize("dtype,V,bounds", [
    (torch.bfloat16, 151936, None),
    (torch.float32, 10007, [0, 513, 6000, 10007]),
])
def test_noalloc_matches_workspace_entry_point_twice(cuda_lib, dtype, V, bounds):
    tol = TOL_FWD[dtype]
    for call, (seed, T) in enumerate([(101, 300), (202, 77)]):
        z, y = _draw(seed, T, V, dtype)
        err = cuda_lib.new_error_flag(z.device)
        lp0, ent0, rs0 = cuda_lib.forward(z, y, IGN, bounds)
        lp1, ent1, rs1 = cuda_lib.forward_noalloc(z, y, IGN, bounds, dev_error=err)
        torch.cuda.synchronize()
        assert err.item() == 0, call
        _same(lp1, lp0, tol)
        _same(ent1, ent0, tol)
        _same(rs1, rs0, tol)
        assert torch.equal(lp1.view(torch.int32), lp0.view(torch.int32)), call


def test_noalloc_refuses_problems_beyond_its_scratch(cuda_lib):
    V = 151936
    chunks = (V + cuda_lib.CHUNK_BF16 - 1) // cuda_lib.CHUNK_BF16
    T = cuda_lib.NOALLOC_SCRATCH_BYTES // (16 * chunks) + 1
    z = torch.empty(T, V, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(T, dtype=torch.int64, device="cuda")
    with pytest.raises(cuda_lib.PstatError) as e:
        cuda_lib.forward_noalloc(z, y)
    assert e.value.code == -6
    # the largest problem that fits is accepted
    Tmax = cuda_lib.NOALLOC_SCRATCH_BYTES // (16 * chunks)
    z2 = (torch.randn(Tmax, V, device="cuda")).to(torch.bfloat16)
    y2 = torch.randint(0, V, (Tmax,), device="cuda")
    lp, ent, rs = cuda_lib.forward_noalloc(z2, y2)
    lp0, ent0, _ = cuda_lib.forward(z2, y2)
    torch.cuda.synchronize()
    assert torch.equal(lp.view(torch.int32), lp0.view(torch.int32))
