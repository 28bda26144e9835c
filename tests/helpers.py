"""Shared test utilities: moving tensors to the oracle and the parity rules.

Tolerances (floating point, per row or element):
  logprob / entropy   |gpu - oracle| <= 1e-5 for fp32 logits, 1e-4 for bf16
                      logits (fp32 accumulation on the GPU), plus two fp32
                      ulps of the oracle value: the outputs are fp32, whose
                      spacing exceeds 1e-5 once |value| > 64;
  dlogits, fp32 out   |g - g*| <= 1e-3 |g*| + 1e-12;
  dlogits, bf16 out   |g - bf16(g*)| <= max(1e-3 |g*|, one bf16 ulp of g*),
                      plus a Frobenius-relative bound 2.5e-3 against g*.
The bf16 rule compares with the correctly rounded exact value because
rounding the exact gradient to bf16 alone already moves it by up to half an
ulp (about 2e-3 relative), more than 1e-3.
"""
import numpy as np
import torch

TOL_FWD = {torch.float32: 1e-5, torch.bfloat16: 1e-4}


def to_oracle(z: torch.Tensor) -> np.ndarray:
    """A CUDA/CPU tensor as the oracle's input array (bf16 as uint16 bits)."""
    z = z.detach().cpu().contiguous()
    if z.dtype == torch.bfloat16:
        return z.view(torch.int16).numpy().view(np.uint16)
    return z.numpy()


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (nearest even) through torch, as float64."""
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).double().numpy()


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (subnormal floor 2^-133)."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.maximum(ax, 2.0**-126)))
    return np.maximum(2.0 ** (e - 7), 2.0**-133)


def assert_forward_close(lp, ent, ref, dtype, rows=None, what=""):
    tol = TOL_FWD[dtype]
    lp = lp.detach().double().cpu().numpy()
    ent = ent.detach().double().cpu().numpy()
    rlp, rent = ref["logprob"], ref["entropy"]
    if rows is not None:
        lp, ent = lp[rows], ent[rows]
    for name, a, b in (("logprob", lp, rlp), ("entropy", ent, rent)):
        both_nan = np.isnan(a) & np.isnan(b)
        both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
        room = tol + 2.0 * np.spacing(np.abs(b).astype(np.float32)).astype(np.float64)
        with np.errstate(invalid="ignore"):  # inf - inf: decided by both_inf
            ok = both_nan | both_inf | (np.abs(a - b) <= room)
        if not ok.all():
            i = int(np.flatnonzero(~ok)[0])
            raise AssertionError(f"{what} {name} row {i}: gpu {a[i]!r} oracle {b[i]!r} "
                                 f"(tol {tol}, {int((~ok).sum())} bad rows)")


def assert_grad_close(g, gref, out_dtype, what=""):
    """g: torch tensor [R, V] from the GPU; gref: float64 oracle [R, V]."""
    a = g.detach().double().cpu().numpy()
    b = np.asarray(gref, np.float64)
    nan_ok = np.isnan(a) & np.isnan(b)
    if out_dtype == torch.float32:
        ok = nan_ok | (np.abs(a - b) <= 1e-3 * np.abs(b) + 1e-12)
    else:
        br = bf16_round(b)
        ok = nan_ok | (np.abs(a - br) <= np.maximum(1e-3 * np.abs(b), bf16_ulp(b)))
        fin = np.isfinite(b)
        den = np.linalg.norm(b[fin])
        if den > 0:
            rel = np.linalg.norm((a - b)[fin]) / den
            assert rel <= 2.5e-3, f"{what} Frobenius-relative {rel}"
    if not ok.all():
        idx = np.argwhere(~ok)[0]
        raise AssertionError(f"{what} dlogits{tuple(idx)}: gpu {a[tuple(idx)]!r} oracle "
                             f"{b[tuple(idx)]!r} ({int((~ok).sum())} bad elements)")


class GradParity:
    """The dlogits rule of ``assert_grad_close`` applied block by block on the
    GPU, for full-size tensors: each block of oracle rows (float64, from the
    CPU oracle) is moved to the device and compared element by element there;
    the Frobenius-relative bound (bf16 outputs) is taken over all blocks."""

    def __init__(self, out_dtype, what=""):
        self.out_dtype = out_dtype
        self.what = what
        self.num = 0.0
        self.den = 0.0
        self.rows = 0

    def add(self, g: torch.Tensor, gref: np.ndarray, row0: int = 0):
        b = torch.from_numpy(np.ascontiguousarray(gref, np.float64)).to(g.device)
        a = g.double()
        nan_ok = torch.isnan(a) & torch.isnan(b)
        if self.out_dtype == torch.float32:
            ok = nan_ok | ((a - b).abs() <= 1e-3 * b.abs() + 1e-12)
        else:
            br = b.to(torch.bfloat16).double()
            # one bf16 ulp at |b|: 2^(floor(log2|b|) - 7), floored at the
            # subnormal spacing 2^-133.  frexp gives |b| = m 2^e, m in [0.5, 1);
            # the power of two is assembled from its float64 bit pattern
            # (exponent field k + 1023), exact on every device.
            _, e = torch.frexp(b.abs().clamp_min(2.0**-126))
            k = e.to(torch.int64) - 8
            ulp = ((k + 1023) << 52).view(torch.float64).clamp_min(2.0**-133)
            ok = nan_ok | ((a - br).abs() <= torch.maximum(1e-3 * b.abs(), ulp))
            fin = torch.isfinite(b)
            self.num += float(((a - b)[fin] ** 2).sum())
            self.den += float((b[fin] ** 2).sum())
        bad = ~ok
        if bool(bad.any()):
            idx = tuple(int(i) for i in torch.nonzero(bad)[0])
            raise AssertionError(
                f"{self.what} dlogits row {row0 + idx[0]} col {idx[1]}: gpu {float(a[idx])!r} "
                f"oracle {float(b[idx])!r} ({int(bad.sum())} bad elements in this block)")
        self.rows += g.shape[0]

    def finish(self):
        if self.out_dtype != torch.float32 and self.den > 0:
            rel = (self.num / self.den) ** 0.5
            assert rel <= 2.5e-3, f"{self.what} Frobenius-relative {rel}"
        return self.rows
