"""Exactly rounded pure-Python restatement for tiny inputs.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Every sum is
``math.fsum`` (correctly rounded), every value a Python float, so the only
errors left are those of ``math.exp``/``math.log``.  It pins the C oracle on
tiny rows; it is far too slow for anything else.

Definitions as in torchtitan PR #4685 ("[RL] Avoid full-vocab gather for TP
policy statistics", Summary and Why): logprob = z_y - logsumexp(z), entropy of
softmax(z), weighted cross-entropy gradient w (onehot(y) - softmax(z)).
"""
from __future__ import annotations

import math


def _lse(row):
    m = max(row)
    if m == -math.inf:
        return math.nan
    return m + math.log(math.fsum(math.exp(x - m) for x in row if x != -math.inf))


def forward_row(row, y, ignore_index=-100):
    """(logprob, entropy) of one row given as a list of Python floats."""
    L = _lse(row)
    if math.isnan(L):
        return math.nan, math.nan
    H = -math.fsum(math.exp(x - L) * (x - L) for x in row if x != -math.inf)
    if y == ignore_index:
        return 0.0, H
    if y < 0 or y >= len(row):
        return math.nan, math.nan
    return row[y] - L, H


def backward_row(row, y, w, ignore_index=-100):
    """Weighted gradient row as a list of floats."""
    if y == ignore_index or w == 0.0:
        return [0.0] * len(row)
    L = _lse(row)
    out = []
    for v, x in enumerate(row):
        p = math.exp(x - L) if x != -math.inf else 0.0
        out.append(w * ((1.0 if v == y else 0.0) - p))
    return out
