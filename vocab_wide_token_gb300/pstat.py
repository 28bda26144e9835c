"""ctypes binding of libpstat.so (argument marshalling only).

Every step of the computation runs in the CUDA kernels behind the C ABI
declared in ``include/pstat.h``; this module turns torch tensors into device
pointers, sizes and the current stream, allocates the workspace with torch,
and raises on a non-zero status.  There is no CPU fallback: importing this
module without a built ``libpstat.so`` raises, and every call needs CUDA
tensors.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpstat.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -m vocab_wide_token_gb300.build` "
        "(nvcc, sm_103a); there is no fallback implementation")

_lib = ctypes.CDLL(LIB_PATH)

# ---- C ABI prototypes -------------------------------------------------------
_i64, _i32, _vp, _sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t


def declare_prototypes(lib: ctypes.CDLL) -> ctypes.CDLL:
    """Set the argument and result types of every entry point of
    include/pstat.h on a loaded copy of the library (ctypes would otherwise
    pass 64-bit sizes as C ints)."""
    lib.pstat_status_string.argtypes = [_i32]
    lib.pstat_status_string.restype = ctypes.c_char_p
    lib.pstat_version.restype = _i32
    lib.pstat_workspace_size.argtypes = [_i64, _i64, _i32, _vp, _i32, ctypes.POINTER(_sz)]
    lib.pstat_workspace_size.restype = _i32
    lib.pstat_forward.argtypes = [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _i32, _vp, _vp, _vp,
                                  _vp, _sz, _vp, _vp]
    lib.pstat_forward.restype = _i32
    lib.pstat_forward_noalloc.argtypes = [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _i32, _vp,
                                          _vp, _vp, _vp, _vp]
    lib.pstat_forward_noalloc.restype = _i32
    lib.pstat_backward.argtypes = [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _i32, _vp,
                                   _i32, _i64, _vp, _sz, _vp, _vp]
    lib.pstat_backward.restype = _i32
    lib.pstat_forward_backward.argtypes = [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _i32,
                                           _vp, _vp, _vp, _vp, _i32, _i64, _vp, _vp]
    lib.pstat_forward_backward.restype = _i32
    lib.pstat_log_softmax.argtypes = [_vp, _i32, _i64, _i64, _i64, _vp, _vp, _i32, _vp, _i32, _i64,
                                      _vp, _sz, _vp, _vp]
    lib.pstat_log_softmax.restype = _i32
    lib.pstat_logprob_diff_metrics.argtypes = [_vp, _vp, _vp, _i64, _i64, _vp, _vp]
    lib.pstat_logprob_diff_metrics.restype = _i32
    lib.pstat_clipped_surrogate.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, ctypes.c_float,
                                            ctypes.c_float, ctypes.c_float, _vp, _vp, _vp]
    lib.pstat_clipped_surrogate.restype = _i32
    lib.pstat_lmhead_workspace_size.argtypes = [_i64, _i64, _i64, ctypes.POINTER(_sz)]
    lib.pstat_lmhead_workspace_size.restype = _i32
    lib.pstat_lmhead_fused.argtypes = [_vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _vp,
                                       _sz, _vp, _vp]
    lib.pstat_lmhead_fused.restype = _i32
    lib.pstat_lmhead_backward.argtypes = [_vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _vp,
                                          _vp, _sz, _vp, _vp]
    lib.pstat_lmhead_backward.restype = _i32
    lib.pstat_shard_stats.argtypes = [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _vp, _vp]
    lib.pstat_shard_stats.restype = _i32
    lib.pstat_combine_shards.argtypes = [_vp, _i64, _i32, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp]
    lib.pstat_combine_shards.restype = _i32
    lib.pstat_backward_shard.argtypes = [_vp, _i32, _i64, _i64, _i64, _vp, _i64, _vp, _vp, _i64,
                                         _i64, _vp, _i32, _i64, _vp, _vp]
    lib.pstat_backward_shard.restype = _i32
    lib.pstat_noalloc_scratch_bytes.argtypes = []
    lib.pstat_noalloc_scratch_bytes.restype = _sz
    lib.pstat_selftest_wait_timeout.argtypes = [ctypes.c_uint64, _vp, _vp]
    lib.pstat_selftest_wait_timeout.restype = _i32
    return lib


declare_prototypes(_lib)

F32, BF16 = 0, 1
OK = 0
ERR = {-1: "NULLPTR", -2: "SHAPE", -3: "SHARDS", -4: "DTYPE", -5: "ALIGN", -6: "WORKSPACE",
       -7: "CUDA", -8: "UNSUPPORTED"}
DEV_BAD_LABEL, DEV_EMPTY_ROW, DEV_TIMEOUT, DEV_RANGE = 0x1, 0x2, 0x4, 0x8
CHUNK_BF16, CHUNK_F32 = 4096, 2048
MAX_SHARDS = 64


class PstatError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = _lib.pstat_status_string(code).decode()
        super().__init__(f"{where}: {ERR.get(code, code)} ({msg})")


def _check(code: int, where: str) -> None:
    if code != OK:
        raise PstatError(code, where)


def _call(dev, where: str, fn, *args) -> None:
    """One ABI call with `dev` current: the library takes the device from
    cudaGetDevice (device properties, per-context set-up, the no-allocation
    scratch), so it must be the device that owns the tensors and the stream."""
    with torch.cuda.device(dev):
        _check(fn(*args), where)


def lib() -> ctypes.CDLL:
    """The loaded C library (for callers that want the raw ABI)."""
    return _lib


def version() -> int:
    return int(_lib.pstat_version())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _rows(logits: torch.Tensor):
    if logits.dim() != 2:
        raise ValueError("logits must be 2-D [T, V]")
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor (no CPU path exists)")
    if logits.stride(1) != 1:
        raise ValueError("logits rows must be contiguous (stride(1) == 1)")
    T, V = logits.shape
    ld = logits.stride(0) if T > 1 else V
    return T, V, ld


def _bounds(shard_bounds, V):
    if shard_bounds is None:
        return None, 1
    b = [int(x) for x in shard_bounds]
    arr = (ctypes.c_int64 * len(b))(*b)
    return arr, len(b) - 1


def _labels(labels, T, device):
    if labels is None:
        return None
    if labels.dtype != torch.int64 or labels.shape != (T,) or labels.device != device:
        raise ValueError("labels must be int64 [T] on the logits' device")
    return labels.contiguous()


# The kernels write through every pointer they get, so a tensor on another
# device, of another size or with gaps would be written out of bounds: the
# checks below reject it before anything is launched.
def _tensor(x, dtype, shape, dev, name):
    if (not isinstance(x, torch.Tensor) or x.dtype != dtype or tuple(x.shape) != tuple(shape)
            or x.device != dev or not x.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous {dtype} tensor of shape {tuple(shape)} "
                         f"on {dev}")
    return x


def _row_outputs(out, T, dev):
    """(logprob [T], entropy [T], rowstats [T, 2]), float32 on `dev`."""
    if out is None:
        return (torch.empty(T, dtype=torch.float32, device=dev),
                torch.empty(T, dtype=torch.float32, device=dev),
                torch.empty(T, 2, dtype=torch.float32, device=dev))
    lp, ent, rs = out
    return (_tensor(lp, torch.float32, (T,), dev, "out[0] (logprob)"),
            _tensor(ent, torch.float32, (T,), dev, "out[1] (entropy)"),
            _tensor(rs, torch.float32, (T, 2), dev, "out[2] (rowstats)"))


def _matrix_output(out, T, V, dev, name):
    """A [T, V] bf16 or fp32 output on `dev` with contiguous rows; returns its row stride."""
    if (out.dim() != 2 or tuple(out.shape) != (T, V) or out.stride(1) != 1
            or out.device != dev or out.dtype not in (torch.bfloat16, torch.float32)
            or (T > 1 and out.stride(0) < V)):
        raise ValueError(f"{name} must be a bf16 or fp32 [T, V] tensor on {dev} "
                         "with contiguous rows")
    return out.stride(0) if T > 1 else V


def _weights(weights, T, dev):
    if weights is None:
        return None
    if weights.dtype != torch.float32 or tuple(weights.shape) != (T,) or weights.device != dev:
        raise ValueError(f"weights must be float32 [T] on {dev}")
    return weights.contiguous()


def _rowstats(rowstats, T, dev):
    if rowstats is None:
        return None
    return _tensor(rowstats, torch.float32, (T, 2), dev, "rowstats")


def _error_flag(flag, dev):
    if flag is None:
        return None
    if (flag.dtype != torch.int32 or flag.numel() < 1 or flag.device != dev
            or not flag.is_contiguous()):
        raise ValueError(f"dev_error must be a contiguous int32 tensor on {dev}")
    return flag


def _workspace(ws, need, dev):
    if ws is None:
        return torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    if ws.dtype != torch.uint8 or ws.device != dev or not ws.is_contiguous():
        raise ValueError(f"workspace must be a contiguous uint8 tensor on {dev}")
    return ws


def workspace_size(T: int, V: int, dtype: torch.dtype, shard_bounds=None) -> int:
    n = ctypes.c_size_t(0)
    arr, ns = _bounds(shard_bounds, V)
    code = BF16 if dtype == torch.bfloat16 else F32
    _check(_lib.pstat_workspace_size(T, V, code, arr, ns, ctypes.byref(n)), "pstat_workspace_size")
    return int(n.value)


# pstat_forward runs as one kernel, with no workspace, up to this many chunks
# per row (include/pstat.h).
FORWARD_ROWS_MAX_CHUNKS = 256


def n_chunks(V: int, dtype: torch.dtype, shard_bounds=None) -> int:
    """Chunks per row of the plan: each shard is cut into whole chunks of
    CHUNK_BF16 / CHUNK_F32 elements from its first column (shape arithmetic
    for sizing only; the library validates the bounds)."""
    c = CHUNK_BF16 if dtype == torch.bfloat16 else CHUNK_F32
    b = [0, int(V)] if shard_bounds is None else [int(x) for x in shard_bounds]
    return sum((b1 - b0 + c - 1) // c for b0, b1 in zip(b[:-1], b[1:]))


def new_error_flag(device) -> torch.Tensor:
    """A device int for the kernels' error bits (PSTAT_DEV_*)."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def forward(logits: torch.Tensor, labels: torch.Tensor | None, ignore_index: int = -100,
            shard_bounds=None, *, out=None, workspace=None, dev_error=None):
    """Per-token logprob, entropy and row statistics (M, ln S).

    Returns (logprob [T] f32, entropy [T] f32, rowstats [T, 2] f32).  `out`
    may supply the three tensors; `workspace` a uint8 CUDA tensor of at least
    ``workspace_size`` bytes.
    """
    T, V, ld = _rows(logits)
    dev = logits.device
    lab = _labels(labels, T, dev)
    lp, ent, rs = _row_outputs(out, T, dev)
    dev_error = _error_flag(dev_error, dev)
    arr, ns = _bounds(shard_bounds, V)
    if workspace is None and n_chunks(V, logits.dtype, shard_bounds) > FORWARD_ROWS_MAX_CHUNKS:
        workspace = _workspace(None, workspace_size(T, V, logits.dtype, shard_bounds), dev)
    elif workspace is not None:
        workspace = _workspace(workspace, 0, dev)
    _call(dev, "pstat_forward", _lib.pstat_forward,
          _ptr(logits), _dtype_code(logits), T, V, ld, _ptr(lab), int(ignore_index), arr, ns,
          _ptr(lp), _ptr(ent), _ptr(rs), _ptr(workspace),
          0 if workspace is None else workspace.numel(), _ptr(dev_error), _stream(dev))
    return lp, ent, rs


NOALLOC_SCRATCH_BYTES = int(_lib.pstat_noalloc_scratch_bytes())


def forward_noalloc(logits: torch.Tensor, labels: torch.Tensor | None, ignore_index: int = -100,
                    shard_bounds=None, *, out=None, dev_error=None):
    """Like ``forward`` but through ``pstat_forward_noalloc``: no workspace is
    passed and the library allocates nothing; its scratch is a fixed
    NOALLOC_SCRATCH_BYTES array inside libpstat.so (T * n_chunks * 16 bytes
    must fit).  For callers that may not allocate device memory at this
    point.  Calls that overlap on the GPU share that scratch and race; keep
    them on one stream."""
    T, V, ld = _rows(logits)
    dev = logits.device
    lab = _labels(labels, T, dev)
    lp, ent, rs = _row_outputs(out, T, dev)
    dev_error = _error_flag(dev_error, dev)
    arr, ns = _bounds(shard_bounds, V)
    _call(dev, "pstat_forward_noalloc", _lib.pstat_forward_noalloc,
          _ptr(logits), _dtype_code(logits), T, V, ld, _ptr(lab), int(ignore_index), arr, ns,
          _ptr(lp), _ptr(ent), _ptr(rs), _ptr(dev_error), _stream(dev))
    return lp, ent, rs


def backward(logits: torch.Tensor, labels: torch.Tensor | None, weights: torch.Tensor | None,
             rowstats: torch.Tensor | None, ignore_index: int = -100, shard_bounds=None,
             out_dtype: torch.dtype | None = None, *, out=None, workspace=None, dev_error=None):
    """dlogits = w (onehot(y) - softmax(z)) as a [T, V] tensor of `out_dtype`
    (default: the logits dtype)."""
    T, V, ld = _rows(logits)
    dev = logits.device
    lab = _labels(labels, T, dev)
    out_dtype = out_dtype or logits.dtype
    if out is None:
        out = torch.empty(T, V, dtype=out_dtype, device=dev)
    ld_out = _matrix_output(out, T, V, dev, "out")
    w = _weights(weights, T, dev)
    rowstats = _rowstats(rowstats, T, dev)
    dev_error = _error_flag(dev_error, dev)
    arr, ns = _bounds(shard_bounds, V)
    ws_ptr, ws_n = None, 0
    if rowstats is None:
        need = workspace_size(T, V, logits.dtype, shard_bounds)
        workspace = _workspace(workspace, need, dev)
        ws_ptr, ws_n = _ptr(workspace), workspace.numel()
    _call(dev, "pstat_backward", _lib.pstat_backward,
          _ptr(logits), _dtype_code(logits), T, V, ld, _ptr(lab), int(ignore_index), _ptr(w),
          _ptr(rowstats), arr, ns, _ptr(out), _dtype_code(out), ld_out, ws_ptr, ws_n,
          _ptr(dev_error), _stream(dev))
    return out


def forward_backward(logits: torch.Tensor, labels: torch.Tensor | None,
                     weights: torch.Tensor | None, ignore_index: int = -100, shard_bounds=None,
                     out_dtype: torch.dtype | None = None, *, out=None, dlogits=None,
                     dev_error=None):
    """pstat_forward and pstat_backward in one pass over the logits (same
    results, bit for bit).  Returns (logprob, entropy, rowstats, dlogits)."""
    T, V, ld = _rows(logits)
    dev = logits.device
    lab = _labels(labels, T, dev)
    out_dtype = out_dtype or logits.dtype
    lp, ent, rs = _row_outputs(out, T, dev)
    if dlogits is None:
        dlogits = torch.empty(T, V, dtype=out_dtype, device=dev)
    ld_out = _matrix_output(dlogits, T, V, dev, "dlogits")
    w = _weights(weights, T, dev)
    dev_error = _error_flag(dev_error, dev)
    arr, ns = _bounds(shard_bounds, V)
    _call(dev, "pstat_forward_backward", _lib.pstat_forward_backward,
          _ptr(logits), _dtype_code(logits), T, V, ld, _ptr(lab), int(ignore_index), _ptr(w), arr,
          ns, _ptr(lp), _ptr(ent), _ptr(rs), _ptr(dlogits), _dtype_code(dlogits), ld_out,
          _ptr(dev_error), _stream(dev))
    return lp, ent, rs, dlogits


# ---- vocabulary-parallel use ---------------------------------------------------
# Each rank holds one vocabulary shard [b_s, b_{s+1}) of every row.  The ranks
# all-gather the [T, 4] shard statistics and fold them in ascending shard
# order, so every rank gets the same bits whatever the collective's algorithm.

def shard_stats(logits: torch.Tensor, labels: torch.Tensor | None, vocab_start: int,
                ignore_index: int = -100, *, out=None, dev_error=None):
    """(M_s, S_s, U_s, z_y) of this vocabulary shard per row, [T, 4] float32;
    labels in the whole vocabulary's numbering (z_y = 0 off the shard)."""
    T, V, ld = _rows(logits)
    dev = logits.device
    lab = _labels(labels, T, dev)
    if out is None:
        out = torch.empty(T, 4, dtype=torch.float32, device=dev)
    out = _tensor(out, torch.float32, (T, 4), dev, "out")
    dev_error = _error_flag(dev_error, dev)
    _call(dev, "pstat_shard_stats", _lib.pstat_shard_stats,
          _ptr(logits), _dtype_code(logits), T, V, ld, _ptr(lab), int(ignore_index),
          int(vocab_start), _ptr(out), _ptr(dev_error), _stream(dev))
    return out


def combine_shards(stats: torch.Tensor, labels: torch.Tensor | None, shard_bounds,
                   ignore_index: int = -100, *, out=None, dev_error=None):
    """Row outputs (logprob, entropy, rowstats) from gathered shard statistics
    stats [T, n_shards, 4], shards in ascending vocabulary order, bounds
    shard_bounds (n_shards + 1 ints from 0 to the vocabulary size)."""
    if (stats.dim() != 3 or stats.shape[2] != 4 or stats.dtype != torch.float32
            or not stats.is_cuda):
        raise ValueError("stats must be a float32 CUDA tensor [T, n_shards, 4]")
    stats = stats.contiguous()
    T, ns = stats.shape[0], stats.shape[1]
    dev = stats.device
    arr, nb = _bounds(shard_bounds, None)
    if nb != ns:
        raise ValueError("shard_bounds must have n_shards + 1 entries")
    lab = _labels(labels, T, dev)
    lp, ent, rs = _row_outputs(out, T, dev)
    dev_error = _error_flag(dev_error, dev)
    _call(dev, "pstat_combine_shards", _lib.pstat_combine_shards,
          _ptr(stats), T, ns, arr, _ptr(lab), int(ignore_index), _ptr(lp), _ptr(ent), _ptr(rs),
          _ptr(dev_error), _stream(dev))
    return lp, ent, rs


def backward_shard(logits: torch.Tensor, labels: torch.Tensor | None,
                   weights: torch.Tensor | None, rowstats: torch.Tensor, vocab_start: int,
                   vocab_total: int, ignore_index: int = -100,
                   out_dtype: torch.dtype | None = None, *, out=None, dev_error=None):
    """dlogits of this vocabulary shard's columns from the global (M, ln S)."""
    T, V, ld = _rows(logits)
    dev = logits.device
    lab = _labels(labels, T, dev)
    out_dtype = out_dtype or logits.dtype
    if out is None:
        out = torch.empty(T, V, dtype=out_dtype, device=dev)
    ld_out = _matrix_output(out, T, V, dev, "out")
    w = _weights(weights, T, dev)
    if rowstats is None:
        raise ValueError("rowstats (the global (M, ln S) per row) is required")
    rowstats = _rowstats(rowstats, T, dev)
    dev_error = _error_flag(dev_error, dev)
    _call(dev, "pstat_backward_shard", _lib.pstat_backward_shard,
          _ptr(logits), _dtype_code(logits), T, V, ld, _ptr(lab), int(ignore_index), _ptr(w),
          _ptr(rowstats), int(vocab_start), int(vocab_total), _ptr(out), _dtype_code(out), ld_out,
          _ptr(dev_error), _stream(dev))
    return out


_side_streams: dict = {}


def _side_stream(device: torch.device, role: str = "h2d") -> torch.cuda.Stream:
    """A stream per device and role, created on first use and kept."""
    s = _side_streams.get((device, role))
    if s is None:
        s = torch.cuda.Stream(device=device)
        _side_streams[(device, role)] = s
    return s


def forward_backward_from_host(logits: torch.Tensor, labels: torch.Tensor | None,
                               weights: torch.Tensor | None, ignore_index: int = -100, *,
                               device=None, out_dtype: torch.dtype | None = None,
                               block_rows: int = 512, out=None, dlogits=None, dev_error=None,
                               dlogits_host: torch.Tensor | None = None):
    """forward_backward on logits, labels and weights that live in host memory
    (pinned, for the copies to run asynchronously).  Row blocks of the logits
    are copied into a double-buffered device staging area on a side stream
    while pstat_forward_backward runs on the previous block on the current
    stream, so after the last copy only one block's kernel remains.  Returns
    device (logprob, entropy, rowstats, dlogits), complete in stream order on
    the current stream.

    With `dlogits_host` (a pinned host [T, V] tensor of the output dtype),
    each block's dlogits is also copied back to it on a second side stream
    as soon as its kernel has run, overlapping the next blocks' copies in and
    kernels; the current stream waits for the last of these copies.

    block_rows: 512 measured best overall on the GB300 host link (T = 8192,
    V = 151,936 bf16): 0.688 M tokens/s with dlogits kept on the device
    (1024: 0.684-0.686, 256: 0.683-0.687) and 0.530-0.533 M with dlogits
    copied back (1024: 0.511-0.513, 256: 0.539), smaller blocks leaving less
    of the first copy in and the last copy out exposed."""
    if logits.is_cuda or logits.dim() != 2 or not logits.is_contiguous():
        raise ValueError("logits must be a contiguous 2-D host tensor")
    T, V = logits.shape
    dev = torch.device(device if device is not None else "cuda")
    if dev.index is None:
        dev = torch.device("cuda", torch.cuda.current_device())
    if block_rows < 1:
        raise ValueError("block_rows must be positive")
    cur = torch.cuda.current_stream(dev)
    side = _side_stream(dev)
    lab = None if labels is None else labels.to(dev, non_blocking=True)
    w = None if weights is None else weights.to(dev, non_blocking=True)
    out_dtype = out_dtype or logits.dtype
    if out is None:
        out = (torch.empty(T, dtype=torch.float32, device=dev),
               torch.empty(T, dtype=torch.float32, device=dev),
               torch.empty(T, 2, dtype=torch.float32, device=dev))
    lp, ent, rs = out
    if dlogits is None:
        dlogits = torch.empty(T, V, dtype=out_dtype, device=dev)
    if dlogits_host is not None and (dlogits_host.is_cuda or dlogits_host.dtype != dlogits.dtype
                                     or tuple(dlogits_host.shape) != (T, V)
                                     or not dlogits_host.is_contiguous()):
        raise ValueError("dlogits_host must be a contiguous host tensor [T, V] of the output dtype")
    if T == 0:
        return lp, ent, rs, dlogits
    back = _side_stream(dev, "d2h") if dlogits_host is not None else None
    B = min(block_rows, T)
    bufs = [torch.empty(B, V, dtype=logits.dtype, device=dev) for _ in range(2)]
    for b in bufs:
        b.record_stream(side)
    start = torch.cuda.Event()
    start.record(cur)
    side.wait_event(start)
    freed = [None, None]  # event: the kernel that last read this buffer has run
    for i, r0 in enumerate(range(0, T, B)):
        r1 = min(T, r0 + B)
        buf = bufs[i % 2][: r1 - r0]
        with torch.cuda.stream(side):
            if freed[i % 2] is not None:
                side.wait_event(freed[i % 2])
            buf.copy_(logits[r0:r1], non_blocking=True)
            copied = torch.cuda.Event()
            copied.record(side)
        cur.wait_event(copied)
        forward_backward(buf, None if lab is None else lab[r0:r1],
                         None if w is None else w[r0:r1], ignore_index,
                         out_dtype=out_dtype, out=(lp[r0:r1], ent[r0:r1], rs[r0:r1]),
                         dlogits=dlogits[r0:r1], dev_error=dev_error)
        freed[i % 2] = torch.cuda.Event()
        freed[i % 2].record(cur)
        if back is not None:
            back.wait_event(freed[i % 2])
            with torch.cuda.stream(back):
                dlogits_host[r0:r1].copy_(dlogits[r0:r1], non_blocking=True)
    if back is not None:
        done = torch.cuda.Event()
        done.record(back)
        cur.wait_event(done)
        dlogits.record_stream(back)
    return lp, ent, rs, dlogits


def log_softmax(logits: torch.Tensor, rowstats: torch.Tensor | None = None, shard_bounds=None,
                out_dtype: torch.dtype | None = None, *, out=None, workspace=None,
                dev_error=None):
    """Every column's log-probability, [T, V] of `out_dtype` (default: the
    logits dtype), from (M, ln S) -- computed first when rowstats is None."""
    T, V, ld = _rows(logits)
    dev = logits.device
    out_dtype = out_dtype or logits.dtype
    if out is None:
        out = torch.empty(T, V, dtype=out_dtype, device=dev)
    ld_out = _matrix_output(out, T, V, dev, "out")
    rowstats = _rowstats(rowstats, T, dev)
    dev_error = _error_flag(dev_error, dev)
    arr, ns = _bounds(shard_bounds, V)
    ws_ptr, ws_n = None, 0
    if rowstats is None:
        need = workspace_size(T, V, logits.dtype, shard_bounds)
        workspace = _workspace(workspace, need, dev)
        ws_ptr, ws_n = _ptr(workspace), workspace.numel()
    _call(dev, "pstat_log_softmax", _lib.pstat_log_softmax,
          _ptr(logits), _dtype_code(logits), T, V, ld, _ptr(rowstats), arr, ns, _ptr(out),
          _dtype_code(out), ld_out, ws_ptr, ws_n, _ptr(dev_error), _stream(dev))
    return out


def _f32_vec(x, T, dev, name):
    if x.dtype != torch.float32 or x.shape != (T,) or x.device != dev:
        raise ValueError(f"{name} must be float32 [T] on the same device")
    return x.contiguous()


def logprob_diff_metrics(logprob, rollout_logprob, labels=None, ignore_index: int = -100):
    """(mean d, mean |d|, max |d|, fraction of bitwise-different tokens) over
    non-ignored tokens, d = logprob - rollout_logprob; a float32 [4] tensor."""
    T = logprob.shape[0]
    dev = logprob.device
    a = _f32_vec(logprob, T, dev, "logprob")
    b = _f32_vec(rollout_logprob, T, dev, "rollout_logprob")
    lab = _labels(labels, T, dev)
    out = torch.empty(4, dtype=torch.float32, device=dev)
    _call(dev, "pstat_logprob_diff_metrics", _lib.pstat_logprob_diff_metrics,
          _ptr(a), _ptr(b), _ptr(lab), int(ignore_index), T, _ptr(out), _stream(dev))
    return out


def clipped_surrogate(logprob, old_logprob, advantages, labels=None, eps_low: float = 0.2,
                      eps_high: float = 0.28, scale: float = 1.0, ignore_index: int = -100):
    """Per-token clipped-ratio loss and its derivative d loss / d logprob
    (the backward's per-token weights).  Returns (loss [T], weight [T])."""
    T = logprob.shape[0]
    dev = logprob.device
    a = _f32_vec(logprob, T, dev, "logprob")
    b = _f32_vec(old_logprob, T, dev, "old_logprob")
    c = _f32_vec(advantages, T, dev, "advantages")
    lab = _labels(labels, T, dev)
    loss = torch.empty(T, dtype=torch.float32, device=dev)
    weight = torch.empty(T, dtype=torch.float32, device=dev)
    _call(dev, "pstat_clipped_surrogate", _lib.pstat_clipped_surrogate,
          _ptr(a), _ptr(b), _ptr(c), _ptr(lab), int(ignore_index), T, float(eps_low),
          float(eps_high), float(scale), _ptr(loss), _ptr(weight), _stream(dev))
    return loss, weight


def lmhead_workspace_size(T: int, V: int, d: int) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.pstat_lmhead_workspace_size(T, V, d, ctypes.byref(n)),
           "pstat_lmhead_workspace_size")
    return int(n.value)


def _lmhead_args(hidden, W):
    if hidden.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise TypeError("hidden and W must be bfloat16")
    if not (hidden.is_cuda and W.is_cuda) or hidden.device != W.device:
        raise ValueError("hidden and W must be CUDA tensors on one device")
    if hidden.dim() != 2 or W.dim() != 2:
        raise ValueError("hidden must be [T, d] and W [V, d]")
    hidden, W = hidden.contiguous(), W.contiguous()
    T, d = hidden.shape
    V, d2 = W.shape
    if d != d2:
        raise ValueError("hidden [T, d] and W [V, d] disagree on d")
    return hidden, W, T, V, d


def lmhead_forward(hidden, W, labels, ignore_index: int = -100, *, workspace=None,
                   dev_error=None):
    """Fused lm_head statistics: logits = hidden W^T never leave the chip."""
    hidden, W, T, V, d = _lmhead_args(hidden, W)
    dev = hidden.device
    lab = _labels(labels, T, dev)
    lp, ent, rs = _row_outputs(None, T, dev)
    dev_error = _error_flag(dev_error, dev)
    workspace = _workspace(workspace, lmhead_workspace_size(T, V, d), dev)
    _call(dev, "pstat_lmhead_fused", _lib.pstat_lmhead_fused,
          _ptr(hidden), _ptr(W), T, V, d, _ptr(lab), int(ignore_index), _ptr(lp), _ptr(ent),
          _ptr(rs), _ptr(workspace), workspace.numel(), _ptr(dev_error), _stream(dev))
    return lp, ent, rs


def lmhead_backward(hidden, W, labels, weights, rowstats, ignore_index: int = -100, *,
                    dhidden=None, dW=None, workspace=None, dev_error=None):
    """Accumulates dhidden += g W and dW += g^T hidden (fp32), g = w (onehot - p)."""
    hidden, W, T, V, d = _lmhead_args(hidden, W)
    dev = hidden.device
    lab = _labels(labels, T, dev)
    if dhidden is None:
        dhidden = torch.zeros(T, d, dtype=torch.float32, device=dev)
    if dW is None:
        dW = torch.zeros(V, d, dtype=torch.float32, device=dev)
    dhidden = _tensor(dhidden, torch.float32, (T, d), dev, "dhidden")
    dW = _tensor(dW, torch.float32, (V, d), dev, "dW")
    w = _weights(weights, T, dev)
    if rowstats is None:
        raise ValueError("rowstats (from lmhead_forward) is required")
    rowstats = _rowstats(rowstats, T, dev)
    dev_error = _error_flag(dev_error, dev)
    workspace = _workspace(workspace, lmhead_workspace_size(T, V, d), dev)
    _call(dev, "pstat_lmhead_backward", _lib.pstat_lmhead_backward,
          _ptr(hidden), _ptr(W), T, V, d, _ptr(lab), int(ignore_index), _ptr(w), _ptr(rowstats),
          _ptr(dhidden), _ptr(dW), _ptr(workspace), workspace.numel(), _ptr(dev_error),
          _stream(dev))
    return dhidden, dW


def selftest_wait_timeout(device, limit_ns: int = 10_000_000) -> int:
    """Runs the library's bounded wait on a barrier that nothing arrives at
    (pstat_selftest_wait_timeout) and returns the device error bits it left:
    PSTAT_DEV_TIMEOUT when the failure path works."""
    dev = torch.device(device)
    flag = new_error_flag(dev)
    _call(dev, "pstat_selftest_wait_timeout", _lib.pstat_selftest_wait_timeout,
          int(limit_ns), _ptr(flag), _stream(dev))
    return int(flag.item())


class PolicyStats(torch.autograd.Function):
    """logprob (differentiable) and entropy (a no-grad metric) of every row.

    Backward folds the incoming logprob gradient into the per-token weights:
    dlogits = grad_logprob_t (onehot(y_t) - softmax(z_t)).
    """

    @staticmethod
    def forward(ctx, logits, labels, ignore_index=-100, shard_bounds=None):
        lp, ent, rs = forward(logits, labels, ignore_index, shard_bounds)
        ctx.save_for_backward(logits, labels, rs)
        ctx.ignore_index = ignore_index
        ctx.mark_non_differentiable(ent)
        return lp, ent

    @staticmethod
    def backward(ctx, grad_lp, grad_ent):
        logits, labels, rs = ctx.saved_tensors
        g = backward(logits, labels, grad_lp.float().contiguous(), rs, ctx.ignore_index)
        return g, None, None, None


def policy_stats(logits, labels, ignore_index: int = -100, shard_bounds=None):
    """Differentiable (logprob, entropy) through the CUDA kernels."""
    return PolicyStats.apply(logits, labels, ignore_index, shard_bounds)


class LmheadPolicyStats(torch.autograd.Function):
    """logprob (differentiable in hidden and W) and entropy (a no-grad metric)
    of every token through the fused lm_head; the logits hidden W^T are never
    materialised.

    Backward: with g = grad_logprob_t (onehot(y_t) - softmax(z_t)), dhidden =
    g W and dW = g^T hidden, accumulated in fp32 by the lm_head backward and
    returned in the dtypes of hidden and W.
    """

    @staticmethod
    def forward(ctx, hidden, W, labels, ignore_index=-100):
        lp, ent, rs = lmhead_forward(hidden, W, labels, ignore_index)
        ctx.save_for_backward(hidden, W, labels, rs)
        ctx.ignore_index = ignore_index
        ctx.mark_non_differentiable(ent)
        return lp, ent

    @staticmethod
    def backward(ctx, grad_lp, grad_ent):
        hidden, W, labels, rs = ctx.saved_tensors
        need_h, need_w = ctx.needs_input_grad[0], ctx.needs_input_grad[1]
        if not (need_h or need_w):
            return None, None, None, None
        dh, dW = lmhead_backward(hidden, W, labels, grad_lp.float().contiguous(), rs,
                                 ctx.ignore_index)
        return (dh.to(hidden.dtype) if need_h else None, dW.to(W.dtype) if need_w else None,
                None, None)


def lmhead_policy_stats(hidden, W, labels, ignore_index: int = -100):
    """Differentiable (logprob, entropy) of hidden W^T through the fused lm_head."""
    return LmheadPolicyStats.apply(hidden, W, labels, ignore_index)
