"""The C-ABI library loads, exports every symbol include/pstat.h declares, and
rejects bad arguments before launching anything.  Runs without a GPU: every
call here fails host-side validation (or, with valid arguments, fails to find
a device), so no kernel is ever launched."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pstat.h")


def _load():
    # PSTAT_TEST_LIB names another build of the library to check (the
    # sanitizer build, see test_abi_sanitized.py).
    path = os.environ.get("PSTAT_TEST_LIB")
    if path:
        from vocab_wide_token_gb300 import pstat

        return pstat.declare_prototypes(ctypes.CDLL(path))
    from vocab_wide_token_gb300 import build

    if not os.path.exists(build.LIB):
        try:
            build.build()
        except RuntimeError as e:  # no nvcc on this machine
            pytest.skip(str(e))
    from vocab_wide_token_gb300 import pstat

    return pstat.lib()


@pytest.fixture(scope="module")
def exports():
    """The library, for symbol and header checks (no calls that launch)."""
    return _load()


@pytest.fixture(scope="module")
def lib():
    """The library, for argument-check calls with made-up device addresses.
    Every call below is meant to fail host-side validation; one that passed
    it would reach device_info, which fails without a GPU.  With a GPU
    present such a call would launch on those addresses, so these tests run
    only where no CUDA device is visible."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("argument checks with made-up device pointers run only without a GPU")
    return _load()


def declared_symbols():
    text = open(HEADER).read()
    return re.findall(r"PSTAT_API\s+[\w\s\*]+?\b(pstat_\w+)\s*\(", text)


def test_header_declares_entry_points():
    names = declared_symbols()
    for must in ("pstat_forward", "pstat_backward", "pstat_lmhead_fused", "pstat_lmhead_backward",
                 "pstat_workspace_size", "pstat_lmhead_workspace_size", "pstat_status_string",
                 "pstat_version"):
        assert must in names


def test_exports_every_declared_symbol(exports):
    for name in declared_symbols():
        assert hasattr(exports, name), f"libpstat.so does not export {name}"


def test_status_strings(lib):
    from vocab_wide_token_gb300 import pstat

    for code in [0, -1, -2, -3, -4, -5, -6, -7, -8, 12345]:
        s = lib.pstat_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert pstat.version() >= 10000


def _fwd(lib, logits=0x1000, dt=1, T=4, V=100, ld=100, bounds=None, ns=1, ws=0x2000,
         ws_bytes=1 << 20, labels=0x3000):
    b = None if bounds is None else (ctypes.c_int64 * len(bounds))(*bounds)
    return lib.pstat_forward(ctypes.c_void_p(logits), dt, T, V, ld, ctypes.c_void_p(labels), -100,
                             b, ns, None, None, None, ctypes.c_void_p(ws), ws_bytes, None, None)


def test_forward_argument_checks(lib):
    assert _fwd(lib, dt=7) == -4                       # dtype
    assert _fwd(lib, V=0) == -2                        # shape
    assert _fwd(lib, ld=99) == -2
    assert _fwd(lib, T=-1) == -2
    assert _fwd(lib, bounds=[0, 50, 40, 100], ns=3) == -3      # not increasing
    assert _fwd(lib, bounds=[1, 50, 100], ns=2) == -3          # not starting at 0
    assert _fwd(lib, bounds=[0, 50, 99], ns=2) == -3           # not ending at V
    assert _fwd(lib, bounds=list(range(0, 66)) + [100], ns=66) == -3  # too many shards
    assert _fwd(lib, T=0, logits=0) == 0               # empty batch is a no-op
    assert _fwd(lib, logits=0) == -1                   # null logits
    assert _fwd(lib, logits=0x1001) == -5              # bf16 logits must be 2-byte aligned
    assert _fwd(lib, labels=0x3004) == -5
    # Up to 256 chunks per row the forward is one kernel and needs no
    # workspace; past that the workspace is required, sized and aligned.
    big = dict(V=4096 * 257, ld=4096 * 257)
    assert _fwd(lib, ws=0, **big) == -6                # no workspace
    assert _fwd(lib, ws_bytes=16, **big) == -6         # workspace too small
    assert _fwd(lib, ws=0x2008, ws_bytes=1 << 30, **big) == -5  # 16-byte aligned workspace


def test_workspace_size(lib):
    n = ctypes.c_size_t(0)
    assert lib.pstat_workspace_size(8192, 151936, 1, None, 1, ctypes.byref(n)) == 0
    # 38 chunks of 4096 per row, 16 bytes each, plus (M, ln S) per row, 256-aligned
    assert n.value >= 8192 * 38 * 16 + 8192 * 8
    b = (ctypes.c_int64 * 4)(0, 50000, 100000, 151936)
    assert lib.pstat_workspace_size(8192, 151936, 1, b, 3, ctypes.byref(n)) == 0
    assert n.value >= 8192 * 39 * 16
    assert lib.pstat_workspace_size(10, 100, 5, None, 1, ctypes.byref(n)) == -4
    assert lib.pstat_workspace_size(10, 100, 0, None, 1, None) == -1


def test_backward_argument_checks(lib):
    def bwd(dt=1, out_dt=1, T=4, V=100, ld=100, ld_out=100, logits=0x1000, out=0x4000,
            rowstats=0x5000, ws=0, ws_bytes=0):
        return lib.pstat_backward(ctypes.c_void_p(logits), dt, T, V, ld, None, -100, None,
                                  ctypes.c_void_p(rowstats), None, 1, ctypes.c_void_p(out), out_dt,
                                  ld_out, ctypes.c_void_p(ws), ws_bytes, None, None)
    assert bwd(dt=1, out_dt=0) == -4       # bf16 logits cannot produce fp32 dlogits
    assert bwd(ld_out=50) == -2
    assert bwd(out=0) == -1
    assert bwd(rowstats=0) == -6           # recompute needs a workspace
    assert bwd(out=0x4001) == -5


def test_forward_backward_argument_checks(lib):
    def fb(dt=1, out_dt=1, T=4, V=100, ld=100, ld_out=100, logits=0x1000, out=0x4000,
           bounds=None, ns=1):
        b = None if bounds is None else (ctypes.c_int64 * len(bounds))(*bounds)
        return lib.pstat_forward_backward(ctypes.c_void_p(logits), dt, T, V, ld, None, -100, None,
                                          b, ns, None, None, None, ctypes.c_void_p(out), out_dt,
                                          ld_out, None, None)
    assert fb(dt=9) == -4
    assert fb(dt=1, out_dt=0) == -4
    assert fb(ld_out=10) == -2
    assert fb(out=0) == -1
    assert fb(logits=0x1001) == -5
    assert fb(T=0, logits=0, out=0) == 0
    # more than 256 chunks per row is refused (records live in shared memory)
    assert fb(V=4096 * 257, ld=4096 * 257, ld_out=4096 * 257) == -2
    assert fb(bounds=[0, 60, 50, 100], ns=3) == -3


def test_noalloc_argument_checks(lib):
    def na(T=4, V=100, logits=0x1000):
        return lib.pstat_forward_noalloc(ctypes.c_void_p(logits), 1, T, V, V, None, -100, None, 1,
                                         None, None, None, None, None)
    assert na(V=0) == -2
    assert na(logits=0) == -1
    assert na(T=0, logits=0) == 0
    # beyond the fixed 8 MiB scratch: 16-byte records per row and chunk
    assert na(T=(8 << 20) // (16 * 38) + 1, V=151936) == -6


def test_lmhead_argument_checks(lib):
    n = ctypes.c_size_t(0)
    assert lib.pstat_lmhead_workspace_size(16384, 151936, 4096, ctypes.byref(n)) == 0
    assert n.value > 16384 * 38 * 16
    assert lib.pstat_lmhead_workspace_size(16, 100, 100, ctypes.byref(n)) == -2   # d % 64
    def fw(h=0x1000, W=0x2000, T=4, V=100, d=128, ws=0x3000, ws_bytes=1 << 20):
        return lib.pstat_lmhead_fused(ctypes.c_void_p(h), ctypes.c_void_p(W), T, V, d, None, -100,
                                      None, None, None, ctypes.c_void_p(ws), ws_bytes, None, None)
    assert fw(d=96) == -2
    assert fw(h=0) == -1
    assert fw(W=0x2008) == -5          # 16-byte alignment for TMA
    assert fw(ws=0) == -6
    assert fw(T=0, h=0, W=0) == 0
    def bw(rowstats=0x5000, dh=0x6000, dW=0x7000, ws=0x8000, ws_bytes=1 << 30):
        return lib.pstat_lmhead_backward(ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), 4, 100,
                                         128, None, -100, None, ctypes.c_void_p(rowstats),
                                         ctypes.c_void_p(dh), ctypes.c_void_p(dW),
                                         ctypes.c_void_p(ws), ws_bytes, None, None)
    assert bw(rowstats=0) == -1        # the backward needs (M, ln S) from the forward
    assert bw(dW=0x7004) == -5
    assert bw(ws_bytes=16) == -6
    assert bw(ws=0x8010) == -5         # 1024-byte aligned workspace


def test_shard_entry_argument_checks(lib):
    c = ctypes.c_void_p
    # pstat_shard_stats(logits, dt, T, V, ld, labels, ignore, vocab_start, out, dev_error, stream)
    def stats(dt=1, T=4, V=100, ld=100, start=0, logits=0x1000, out=0x2000):
        return lib.pstat_shard_stats(c(logits), dt, T, V, ld, None, -100, start, c(out), None,
                                     None)
    assert stats(dt=7) == -4
    assert stats(V=0) == -2
    assert stats(ld=50) == -2
    assert stats(start=-1) == -2
    assert stats(V=256 * 4096 + 1, ld=256 * 4096 + 1) == -2  # more than 256 chunks
    assert stats(T=0) == 0
    assert stats(out=0) == -1
    assert stats(out=0x2008) == -5                             # float4 output: 16-byte aligned
    # pstat_combine_shards(stats, T, n_shards, bounds, labels, ignore, lp, ent, rs, err, stream)
    def comb(bounds, n=None, T=4, st=0x3000):
        b = (ctypes.c_int64 * len(bounds))(*bounds)
        n = len(bounds) - 1 if n is None else n
        return lib.pstat_combine_shards(c(st), T, n, b, None, -100, None, None, None, None,
                                        None)
    assert comb([0, 10, 5]) == -3
    assert comb([1, 10]) == -3
    assert comb([0, 10], n=0) == -3
    assert comb([0, 10], T=-1) == -2
    assert comb([0, 10], T=0) == 0
    assert comb([0, 10], st=0) == -1
    assert comb([0, 10], st=0x3004) == -5
    # pstat_backward_shard(logits, dt, T, V, ld, labels, ignore, w, rs, start, total, out,
    #                      out_dt, ld_out, err, stream)
    def bwd(dt=1, out_dt=1, V=100, start=0, total=100, rs=0x4000):
        return lib.pstat_backward_shard(c(0x1000), dt, 4, V, V, None, -100, None, c(rs), start,
                                        total, c(0x5000), out_dt, V, None, None)
    assert bwd(dt=1, out_dt=0) == -4
    assert bwd(start=50, total=120) == -2
    assert bwd(rs=0) == -1


def test_binding_rejects_tensors_the_kernels_would_overrun(lib):
    """The Python layer checks every tensor it hands to a kernel (dtype,
    shape, device, layout) and raises before any launch.  The checks compare
    devices only, so they run here against the CPU device."""
    import torch

    from vocab_wide_token_gb300 import pstat

    cpu, T, V = torch.device("cpu"), 5, 7
    f32 = torch.float32
    # row outputs: right ones pass, a short or mistyped one does not
    ok = (torch.empty(T), torch.empty(T), torch.empty(T, 2))
    assert all(a is b for a, b in zip(pstat._row_outputs(ok, T, cpu), ok))
    for bad in ((torch.empty(T - 1), ok[1], ok[2]), (ok[0], ok[1].double(), ok[2]),
                (ok[0], ok[1], torch.empty(T, 3)), (ok[0], ok[1], torch.empty(2, T).t())):
        with pytest.raises(ValueError):
            pstat._row_outputs(bad, T, cpu)
    # outputs on another device
    with pytest.raises(ValueError):
        pstat._row_outputs(ok, T, torch.device("cuda", 0))
    # [T, V] outputs: rows may be padded, not overlap or be strided
    big = torch.empty(T, V + 3, dtype=torch.bfloat16)
    assert pstat._matrix_output(big[:, :V], T, V, cpu, "out") == V + 3
    for bad in (torch.empty(T, V, dtype=torch.float16), torch.empty(V, T).t(),
                torch.empty(T, V + 1)[:, 1:].as_strided((T, V), (V - 1, 1)),
                torch.empty(T + 1, V)):
        with pytest.raises(ValueError):
            pstat._matrix_output(bad, T, V, cpu, "out")
    with pytest.raises(ValueError):
        pstat._weights(torch.empty(T, dtype=torch.float64), T, cpu)
    with pytest.raises(ValueError):
        pstat._rowstats(torch.empty(T, 2, dtype=f32).t().contiguous().t(), T, cpu)
    with pytest.raises(ValueError):
        pstat._error_flag(torch.zeros(1, dtype=torch.int64), cpu)
    with pytest.raises(ValueError):
        pstat._workspace(torch.empty(64, dtype=f32), 16, cpu)
    assert pstat._workspace(None, 100, cpu).numel() == 100
    assert pstat._rowstats(None, T, cpu) is None and pstat._weights(None, T, cpu) is None


def test_noalloc_scratch_size_matches_header(exports):
    # The binding sizes its checks from the library's exported value; both
    # must agree with the header's PSTAT_NOALLOC_SCRATCH_BYTES.
    from vocab_wide_token_gb300 import pstat

    m = re.search(r"#define PSTAT_NOALLOC_SCRATCH_BYTES \((\d+)u << (\d+)\)", open(HEADER).read())
    want = int(m.group(1)) << int(m.group(2))
    exports.pstat_noalloc_scratch_bytes.restype = ctypes.c_size_t
    assert exports.pstat_noalloc_scratch_bytes() == want == pstat.NOALLOC_SCRATCH_BYTES


def test_selftest_argument_checks(lib):
    # the device error flag is required; the wait limit is at most one second
    assert lib.pstat_selftest_wait_timeout(1000, None, None) == -1
    assert lib.pstat_selftest_wait_timeout(2_000_000_000, ctypes.c_void_p(0x1000), None) == -2
