"""Float64 oracle for the fused lm_head variant.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The fused path never materialises logits, but what it computes is plainly
defined: logits z = h W^T from the bfloat16 hidden states h [T, d] and the
bfloat16 vocabulary projection W [V, d] (the chunked lm_head multiply of TRL
PR #6949 "ZeroSyncGRPOTrainer"), followed by the same per-token statistics as
the unfused path.  The backward is the chain rule through z = h W^T of the
weighted gradient g = w (onehot(y) - softmax(z)):
    dhidden = g W,    dW = g^T h.
The lm_head backward on that page keeps its GEMMs in the model dtype and
accumulates in fp32; here every product is float64 (numpy matmul, a library
primitive), so the oracle is the exact target those roundings approximate.
"""
from __future__ import annotations

import numpy as np

from . import backward as _backward
from . import bf16_to_f64
from . import forward as _forward


def _f64(x: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) or a float array, widened to float64."""
    x = np.asarray(x)
    return bf16_to_f64(x) if x.dtype == np.uint16 else x.astype(np.float64)


def logits(h_bits: np.ndarray, W_bits: np.ndarray, rows=None) -> np.ndarray:
    """z = h W^T in float64; optional row subset of h."""
    h = _f64(h_bits if rows is None else np.asarray(h_bits)[rows])
    return h @ _f64(W_bits).T


def forward(h_bits, W_bits, labels, ignore_index=-100, rows=None):
    z = logits(h_bits, W_bits, rows)
    lab = np.asarray(labels, np.int64)
    if rows is not None:
        lab = lab[rows]
    return _forward(z, lab, ignore_index)


def backward(h_bits, W_bits, labels, weights, ignore_index=-100):
    """Returns (dhidden [T, d], dW [V, d]) in float64 over all T rows."""
    h = _f64(h_bits)
    W = _f64(W_bits)
    z = h @ W.T
    g = _backward(z, np.asarray(labels, np.int64), np.asarray(weights, np.float64), ignore_index)
    return g @ W, g.T @ h
