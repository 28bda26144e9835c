"""pstat_forward_noalloc: the forward statistics for callers that cannot
allocate device memory (allocation would synchronise the device, or their
host owns all device memory through its own pool, or they have no allocator).

It takes no workspace; its scratch is a fixed array inside libpstat.so.  The
test calls it through the C ABI (ctypes binding) twice in a row on different
inputs and checks each result against the workspace entry point pstat_forward
with the parity tolerances the other tests use (the kernels are the same, so
the results are in fact expected to be identical bit for bit), checks that
a problem larger than the fixed scratch is refused before any launch, and
that calls keep working after cudaDeviceReset (the scratch's address is
looked up again in the new context).

This file is named so that pytest collects it last."""
import os
import subprocess
import sys

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


# Runs in a fresh process that uses only ctypes: libpstat.so and the CUDA
# runtime it links (the same loaded copy), no torch.  Each round allocates its
# buffers with cudaMalloc (the test may allocate; the entry point under test
# does not), compares pstat_forward_noalloc with pstat_forward bit for bit,
# and the second round runs after cudaDeviceReset, which ends this process's
# context: the library must look the scratch address and the kernels'
# shared-memory opt-ins up again in the new context.
_RESET_SCRIPT = r"""
import ctypes, sys
import numpy as np
lib = ctypes.CDLL(sys.argv[1])
rt = ctypes.CDLL("libcudart.so.13")
vp, i64, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
rt.cudaMalloc.argtypes = [ctypes.POINTER(vp), sz]
rt.cudaMemcpy.argtypes = [vp, vp, sz, ctypes.c_int]
rt.cudaMemset.argtypes = [vp, ctypes.c_int, sz]
rt.cudaFree.argtypes = [vp]
lib.pstat_forward.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, i64, vp, ctypes.c_int, vp, vp,
                              vp, vp, sz, vp, vp]
lib.pstat_forward_noalloc.argtypes = [vp, ctypes.c_int, i64, i64, i64, vp, i64, vp, ctypes.c_int,
                                      vp, vp, vp, vp, vp]
lib.pstat_workspace_size.argtypes = [i64, i64, ctypes.c_int, vp, ctypes.c_int, ctypes.POINTER(sz)]

def ok(rc, what):
    if rc != 0:
        raise SystemExit(f"{what} returned {rc}")

def dev_buf(nbytes, host=None):
    p = vp()
    ok(rt.cudaMalloc(ctypes.byref(p), max(nbytes, 16)), "cudaMalloc")
    if host is not None:
        ok(rt.cudaMemcpy(p, host.ctypes.data, nbytes, 1), "cudaMemcpy H2D")
    return p

def one_round(seed):
    T, V = 257, 10007
    bounds = (i64 * 4)(0, 513, 6000, V)
    rng = np.random.default_rng(seed)
    z = (2.0 * rng.standard_normal((T, V))).astype(np.float32)
    y = rng.integers(0, V, T).astype(np.int64)
    y[1] = -100
    n = sz(0)
    ok(lib.pstat_workspace_size(T, V, 0, bounds, 3, ctypes.byref(n)), "pstat_workspace_size")
    dz, dy = dev_buf(z.nbytes, z), dev_buf(y.nbytes, y)
    ws, err = dev_buf(n.value), dev_buf(4)
    ok(rt.cudaMemset(err, 0, 4), "cudaMemset")
    outs = [[dev_buf(4 * T), dev_buf(4 * T), dev_buf(8 * T)] for _ in range(2)]
    ok(lib.pstat_forward(dz, 0, T, V, V, dy, -100, bounds, 3, *outs[0], ws, n.value, err, None),
       "pstat_forward")
    ok(lib.pstat_forward_noalloc(dz, 0, T, V, V, dy, -100, bounds, 3, *outs[1], err, None),
       "pstat_forward_noalloc")
    ok(rt.cudaDeviceSynchronize(), "cudaDeviceSynchronize")
    host = []
    for o in outs:
        hs = [np.empty(T, np.float32), np.empty(T, np.float32), np.empty((T, 2), np.float32)]
        for h, d in zip(hs, o):
            ok(rt.cudaMemcpy(h.ctypes.data, d, h.nbytes, 2), "cudaMemcpy D2H")
        host.append(hs)
    e = np.zeros(1, np.int32)
    ok(rt.cudaMemcpy(e.ctypes.data, err, 4, 2), "cudaMemcpy D2H")
    if e[0] != 0:
        raise SystemExit(f"device error bits {e[0]}")
    for a, b, name in zip(host[0], host[1], ("logprob", "entropy", "rowstats")):
        if not np.array_equal(a.view(np.int32), b.view(np.int32)):
            raise SystemExit(f"round {seed}: {name} differs from pstat_forward")
    if not np.all(np.isfinite(host[1][0][y != -100])):
        raise SystemExit("non-finite logprob")
    for p in [dz, dy, ws, err] + outs[0] + outs[1]:
        rt.cudaFree(p)

ok(rt.cudaSetDevice(0), "cudaSetDevice")
one_round(1)
ok(rt.cudaDeviceReset(), "cudaDeviceReset")
one_round(2)
print("ok")
"""


def test_noalloc_after_device_reset(cuda_lib):
    r = subprocess.run([sys.executable, "-c", _RESET_SCRIPT, cuda_lib.LIB_PATH],
                       capture_output=True, text=True, timeout=300,
                       env={**os.environ, "CUDA_VISIBLE_DEVICES": os.environ.get(
                           "CUDA_VISIBLE_DEVICES", "0")})
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr


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
