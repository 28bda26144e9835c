"""Float64 oracle for the loss-side epilogue of the policy statistics.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

1. Trainer/rollout mismatch metrics, as the torchtitan batch-invariant GDN
   README logs them ("Code map": ``bit_wise/logprob_diff/{mean,abs_mean,max}``
   and ``bit_wise/ratio_tokens_different/mean``, between the trainer's
   recomputed logprob pi and the generator's rollout logprob mu).  Over the
   tokens whose label is not the ignore index, with d_t = pi_t - mu_t:
       mean      = sum_t d_t / n
       abs_mean  = sum_t |d_t| / n
       max       = max_t |d_t|      (the largest mismatch, in absolute value)
       different = (number of tokens whose float32 bit patterns differ) / n
   With n = 0 the means and the ratio are NaN and the max is 0.

2. The clipped-ratio surrogate of the same README's DAPO recipes (clip
   (0.2, 0.28)): per token, r_t = exp(pi_t - pi_old_t),
       loss_t = -scale * min(r_t A_t, clip(r_t, 1 - eps_low, 1 + eps_high) A_t)
   and its derivative with respect to pi_t, which is the weight the
   logprob backward multiplies (onehot - softmax) by:
       dloss_t/dpi_t = -scale * A_t * r_t   when the unclipped term is the
                                             smaller one (or they tie),
                     = 0                     when the clipped term is smaller
                                             (it does not depend on pi_t).
   Ignored tokens have loss 0 and weight 0.
"""
from __future__ import annotations

import math

import numpy as np


def diff_metrics(pi, mu, labels, ignore_index=-100):
    pi = np.asarray(pi, np.float32)
    mu = np.asarray(mu, np.float32)
    keep = np.asarray(labels) != ignore_index
    n = int(keep.sum())
    if n == 0:
        return {"mean": math.nan, "abs_mean": math.nan, "max": 0.0, "different": math.nan}
    d = pi[keep].astype(np.float64) - mu[keep].astype(np.float64)
    differ = pi[keep].view(np.uint32) != mu[keep].view(np.uint32)
    return {"mean": math.fsum(d) / n, "abs_mean": math.fsum(np.abs(d)) / n,
            "max": float(np.max(np.abs(d))), "different": float(differ.sum()) / n}


def clipped_surrogate(pi, pi_old, adv, labels, eps_low=0.2, eps_high=0.28, scale=1.0,
                      ignore_index=-100):
    """Returns (loss [T], weight [T]) in float64."""
    pi = np.asarray(pi, np.float64)
    pi_old = np.asarray(pi_old, np.float64)
    adv = np.asarray(adv, np.float64)
    keep = np.asarray(labels) != ignore_index
    T = pi.shape[0]
    loss = np.zeros(T)
    weight = np.zeros(T)
    for t in range(T):
        if not keep[t]:
            continue
        r = math.exp(pi[t] - pi_old[t])
        rc = min(max(r, 1.0 - eps_low), 1.0 + eps_high)
        unclipped, clipped = r * adv[t], rc * adv[t]
        if unclipped <= clipped:
            loss[t] = -scale * unclipped
            weight[t] = -scale * adv[t] * r
        else:
            loss[t] = -scale * clipped
            weight[t] = 0.0
    return loss, weight
