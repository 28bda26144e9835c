"""Float64 CPU oracle for per-token policy statistics.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``vocab_wide_token_gb300``) never imports it and has no CPU fallback.

The arithmetic lives in ``pstat_oracle.c`` (plain C, double precision, OpenMP
over rows); this module only builds it with gcc on first use and marshals numpy
arrays.  ``lmhead`` adds the fused-lm_head oracle (numpy float64 matmul then
the same C routines) and ``bruteforce`` an exactly rounded pure-Python version
for tiny inputs.

Sources followed (torchtitan PR #4685, "[RL] Avoid full-vocab gather for TP
policy statistics"): Summary and Why (global maximum, softmax denominator,
target contribution, entropy-weighted sum; entropy is a no-grad metric),
Correctness and compatibility (ignored labels, partially masked logits,
uneven vocabulary shards, weighted gradients), and the review diff that writes
logprobs as the negated cross entropy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pstat_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, BF16, F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile ``pstat_oracle.c`` into ``liboracle.so`` (gcc, OpenMP)."""
    with _lock:
        stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                   "-o", tmp, _SRC, "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        # ORACLE_LIB names a prebuilt copy; the mutation test uses it to load
        # deliberately broken builds of pstat_oracle.c.
        path = os.environ.get("ORACLE_LIB") or build()
        lib = ctypes.CDLL(path)
        i64, vp, dp, i = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int
        lib.oracle_forward.argtypes = [vp, i, i64, i64, i64, vp, i64, dp, dp, dp, dp]
        lib.oracle_forward.restype = i
        lib.oracle_backward.argtypes = [vp, i, i64, i64, i64, vp, i64, dp, dp]
        lib.oracle_backward.restype = i
        lib.oracle_sharded.argtypes = [vp, i, i64, i64, i64, vp, i64, vp, i, dp, dp, dp]
        lib.oracle_sharded.restype = i
        lib.oracle_set_threads.argtypes = [i]
        lib.oracle_threads.restype = i
        _lib = lib
    return _lib


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def threads() -> int:
    return int(_load().oracle_threads())


def _as_logits(z):
    """Return (contiguous 2-D array, dtype code, ld).  bfloat16 is passed as
    uint16 bit patterns (see ``bf16_bits``)."""
    z = np.asarray(z)
    if z.ndim != 2:
        raise ValueError("logits must be 2-D [T, V]")
    if z.dtype == np.float32:
        code = F32
    elif z.dtype == np.uint16:
        code = BF16
    elif z.dtype == np.float64:
        code = F64
    else:
        raise TypeError(f"unsupported logits dtype {z.dtype}")
    z = np.ascontiguousarray(z)
    return z, code, z.shape[1]


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _labels(labels, T):
    if labels is None:
        return None
    lab = np.ascontiguousarray(np.asarray(labels, dtype=np.int64))
    if lab.shape != (T,):
        raise ValueError("labels must be [T]")
    return lab


def forward(z, labels, ignore_index=-100):
    """Returns dict(logprob, entropy, M, logS), each float64 [T]."""
    z, code, ld = _as_logits(z)
    T, V = z.shape
    lab = _labels(labels, T)
    out = {k: np.empty(T, np.float64) for k in ("logprob", "entropy", "M", "logS")}
    rc = _load().oracle_forward(_ptr(z), code, T, V, ld, _ptr(lab), int(ignore_index),
                                _ptr(out["logprob"]), _ptr(out["entropy"]),
                                _ptr(out["M"]), _ptr(out["logS"]))
    if rc != 0:
        raise ValueError("oracle_forward rejected its arguments")
    return out


def backward(z, labels, weights=None, ignore_index=-100):
    """Returns dlogits float64 [T, V] = w (onehot(y) - softmax(z))."""
    z, code, ld = _as_logits(z)
    T, V = z.shape
    lab = _labels(labels, T)
    w = None if weights is None else np.ascontiguousarray(np.asarray(weights, np.float64))
    out = np.empty((T, V), np.float64)
    rc = _load().oracle_backward(_ptr(z), code, T, V, ld, _ptr(lab), int(ignore_index),
                                 _ptr(w), _ptr(out))
    if rc != 0:
        raise ValueError("oracle_backward rejected its arguments")
    return out


def log_softmax(z):
    """log softmax of every row, float64 [T, V]: z - (M + ln S) with (M, ln S)
    from ``forward`` (the log-partition of the plain definition)."""
    zz, code, ld = _as_logits(z)
    st = forward(zz, None)
    if code == BF16:
        z64 = bf16_to_f64(zz)
    else:
        z64 = zz.astype(np.float64)
    return z64 - (st["M"] + st["logS"])[:, None]


def sharded(z, labels, bounds, ignore_index=-100):
    """Shard-local (m, s, u) [T, n_shards, 3] and the combined logprob/entropy."""
    z, code, ld = _as_logits(z)
    T, V = z.shape
    lab = _labels(labels, T)
    b = np.ascontiguousarray(np.asarray(bounds, np.int64))
    ns = len(b) - 1
    stats = np.empty((T, ns, 3), np.float64)
    lp = np.empty(T, np.float64)
    H = np.empty(T, np.float64)
    rc = _load().oracle_sharded(_ptr(z), code, T, V, ld, _ptr(lab), int(ignore_index),
                                _ptr(b), ns, _ptr(stats), _ptr(lp), _ptr(H))
    if rc != 0:
        raise ValueError("oracle_sharded rejected its arguments")
    return {"shard_stats": stats, "logprob": lp, "entropy": H}


def bf16_bits(x_f32: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest even) and return the
    16-bit patterns.  Used only to build oracle-side test inputs."""
    a = np.ascontiguousarray(np.asarray(x_f32, np.float32)).view(np.uint32)
    nan = (a & 0x7FFFFFFF) > 0x7F800000
    rounded = (a + 0x7FFF + ((a >> 16) & 1)) >> 16
    out = np.where(nan, (a >> 16) | 0x40, rounded).astype(np.uint16)
    return out


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
