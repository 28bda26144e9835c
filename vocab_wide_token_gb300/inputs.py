"""Seeded synthetic workloads (no arithmetic of the method itself).

Both the CUDA path and the oracle are fed from here; nothing in this module
computes a logprob, an entropy, a softmax statistic or a gradient.  Labels are
drawn from each row's softmax with the Gumbel-max trick (argmax of logits plus
Gumbel noise), which samples a class without normalising anything.

Workloads (vocabulary of the Qwen3 tokenizer, V = 151,936, as in the pages'
component benchmark):
  tiny     T=64,   V=1000,   fp32 N(0, 3^2), uniform labels with 5 ignored,
           shards {0, 512, 1000}, weights N(0, 1)
  forward  T=4096, V=151936, bf16 N(0, 2^2) with 10% of rows given one
           column +15 (peaked), labels sampled from the row's softmax
  fwdbwd   T=8192, V=151936, bf16 N(0, 2^2), sampled labels, weights
           N(0, 1) advantage times a 0/1 mask with 20% zeros
  uneven   T=8192, V=151936, shards {0, 50000, 100000, 151936}, N(0, 2^2)
           in fp32 or bf16, 25% of rows with 10% of their columns at -inf,
           5% ignored labels, the rest sampled from the masked row
  lmhead   hidden [16384, 4096] bf16 N(0, 1), W [151936, 4096] bf16
           N(0, 0.02^2), labels sampled from softmax(hidden W^T),
           weights N(0, 1)
Every generator takes the seed, the sizes and the device, so tests can draw
smaller instances of the same law.
"""
from __future__ import annotations

import math

import torch

V_QWEN3 = 151936
IGNORE_INDEX = -100


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def gumbel_max(z: torch.Tensor, g: torch.Generator, block: int = 1024) -> torch.Tensor:
    """Labels y_t = argmax_v (z_tv + G_tv), G ~ Gumbel(0, 1), in fp32.
    -inf logits are never chosen while a row has a finite entry."""
    T = z.shape[0]
    out = torch.empty(T, dtype=torch.int64, device=z.device)
    tiny = torch.finfo(torch.float32).tiny
    for r0 in range(0, T, block):
        zz = z[r0:r0 + block].float()
        u = torch.rand(zz.shape, generator=g, device=z.device, dtype=torch.float32)
        gum = -torch.log(-torch.log(u.clamp_(min=tiny)))
        out[r0:r0 + block] = torch.argmax(zz + gum, dim=1)
    return out


def tiny(seed: int = 0, device="cpu", T: int = 64, V: int = 1000, n_ignored: int = 5):
    g = _gen(seed, device)
    z = 3.0 * torch.randn(T, V, generator=g, device=device, dtype=torch.float32)
    y = torch.randint(0, V, (T,), generator=g, device=device, dtype=torch.int64)
    y[torch.randperm(T, generator=g, device=device)[:n_ignored]] = IGNORE_INDEX
    w = torch.randn(T, generator=g, device=device, dtype=torch.float32)
    return {"logits": z, "labels": y, "weights": w, "shard_bounds": [0, 512, V] if V > 512 else None}


def forward_workload(seed: int = 1, device="cpu", T: int = 4096, V: int = V_QWEN3,
                     peak_frac: float = 0.1, peak: float = 15.0, dtype=torch.bfloat16):
    g = _gen(seed, device)
    z = 2.0 * torch.randn(T, V, generator=g, device=device, dtype=torch.float32)
    n_peak = int(round(peak_frac * T))
    rows = torch.randperm(T, generator=g, device=device)[:n_peak]
    cols = torch.randint(0, V, (n_peak,), generator=g, device=device)
    z[rows, cols] += peak
    z = z.to(dtype)
    y = gumbel_max(z, g)
    return {"logits": z, "labels": y, "peaked_rows": rows}


def fwdbwd_workload(seed: int = 2, device="cpu", T: int = 8192, V: int = V_QWEN3,
                    zero_frac: float = 0.2, dtype=torch.bfloat16):
    g = _gen(seed, device)
    z = (2.0 * torch.randn(T, V, generator=g, device=device, dtype=torch.float32)).to(dtype)
    y = gumbel_max(z, g)
    adv = torch.randn(T, generator=g, device=device, dtype=torch.float32)
    keep = (torch.rand(T, generator=g, device=device) >= zero_frac).float()
    return {"logits": z, "labels": y, "weights": adv * keep}


def uneven_workload(seed: int = 3, device="cpu", T: int = 8192, V: int = V_QWEN3,
                    bounds=(0, 50000, 100000, V_QWEN3), dtype=torch.bfloat16,
                    masked_row_frac: float = 0.25, masked_col_frac: float = 0.1,
                    ignored_frac: float = 0.05):
    g = _gen(seed, device)
    z = 2.0 * torch.randn(T, V, generator=g, device=device, dtype=torch.float32)
    n_rows = int(round(masked_row_frac * T))
    n_cols = int(round(masked_col_frac * V))
    rows = torch.randperm(T, generator=g, device=device)[:n_rows]
    for r0 in range(0, n_rows, 256):
        rr = rows[r0:r0 + 256]
        keys = torch.rand(len(rr), V, generator=g, device=device)
        cols = torch.argsort(keys, dim=1)[:, :n_cols]
        sub = z[rr]
        sub.scatter_(1, cols, -math.inf)
        z[rr] = sub
    z = z.to(dtype)
    y = gumbel_max(z, g)
    n_ign = int(round(ignored_frac * T))
    y[torch.randperm(T, generator=g, device=device)[:n_ign]] = IGNORE_INDEX
    b = list(bounds)
    if b[-1] != V:
        b[-1] = V
    return {"logits": z, "labels": y, "shard_bounds": b, "masked_rows": rows}


def lmhead_workload(seed: int = 4, device="cpu", T: int = 16384, V: int = V_QWEN3,
                    d: int = 4096, w_std: float = 0.02, label_block: int = 1024):
    g = _gen(seed, device)
    h = torch.randn(T, d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    W = (w_std * torch.randn(V, d, generator=g, device=device, dtype=torch.float32)).to(torch.bfloat16)
    # Labels from softmax(h W^T): logits are formed block by block with a
    # bf16 matmul for sampling only; they are discarded afterwards.
    y = torch.empty(T, dtype=torch.int64, device=device)
    for r0 in range(0, T, label_block):
        zb = h[r0:r0 + label_block] @ W.t()
        y[r0:r0 + label_block] = gumbel_max(zb, g)
        del zb
    w = torch.randn(T, generator=g, device=device, dtype=torch.float32)
    return {"hidden": h, "W": W, "labels": y, "weights": w}
