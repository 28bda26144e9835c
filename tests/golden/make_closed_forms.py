"""Write ``closed_forms.txt``: closed-form logprob/entropy values at 40 digits.

The values come from the closed forms of the softmax over rows with at most
two distinct finite values, evaluated with Python's ``decimal`` module.  This
script calls nothing in ``oracle/`` and nothing in the CUDA package: it is an
independent pin for both.

Definitions (torchtitan PR #4685, "[RL] Avoid full-vocab gather for TP policy
statistics", Summary; logprob is the negated cross entropy per its review
diff; natural logarithms):
  a row with k entries equal to a and V - k entries equal to b has
    Z  = k e^a + (V - k) e^b
    logprob at an a-entry = a - ln Z,  at a b-entry = b - ln Z
    entropy = ln Z - (k a e^a + (V - k) b e^b) / Z
  k = V (or a = b) is the uniform row: logprob = -ln V, entropy = ln V.
"""
from __future__ import annotations

import os
from decimal import Decimal, getcontext

getcontext().prec = 120

# (name, V, k, a, b); a and b are exactly representable in bfloat16 and float32.
CASES = [
    ("uniform_V1000", 1000, 1000, "0", "0"),
    ("uniform_V151936", 151936, 151936, "0", "0"),
    ("uniform_V151936_shift", 151936, 151936, "3.5", "3.5"),
    ("uniform_V7", 7, 7, "-2", "-2"),
    ("uniform_V1001", 1001, 1001, "1.25", "1.25"),
    ("twolevel_V1000_k1", 1000, 1, "5", "0"),
    ("twolevel_V1000_k500", 1000, 500, "1", "-1"),
    ("twolevel_V151936_k10", 151936, 10, "7.25", "-1.5"),
    ("twolevel_V151936_k1_peak15", 151936, 1, "15", "0"),
    ("nearonehot_V151936_peak100", 151936, 1, "100", "0"),
    ("twolevel_V8_k3", 8, 3, "0.5", "-0.75"),
]


def closed_form(V, k, a, b):
    V, k, a, b = Decimal(V), Decimal(k), Decimal(a), Decimal(b)
    ea, eb = a.exp(), b.exp()
    Z = k * ea + (V - k) * eb
    lnZ = Z.ln()
    H = lnZ - (k * a * ea + (V - k) * b * eb) / Z
    return a - lnZ, b - lnZ, H


def main():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_forms.txt")
    lines = [
        "# Closed-form per-token statistics of two-level rows (natural log).",
        "# Source: softmax definitions of torchtitan PR #4685 '[RL] Avoid full-vocab",
        "# gather for TP policy statistics' (Summary; logprob = -cross_entropy per its",
        "# review diff).  Written by make_closed_forms.py with decimal at 120 digits.",
        "# columns: name V k a b logprob_at_a logprob_at_b entropy",
    ]
    for name, V, k, a, b in CASES:
        lpa, lpb, H = closed_form(V, k, a, b)
        lines.append(f"{name} {V} {k} {a} {b} {lpa:.40e} {lpb:.40e} {H:.40e}")
    with open(path, "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
