"""Pins for the float64 oracle, against things other than the oracle itself.

Each test ties the oracle to mathematics or to an independent routine: closed
forms evaluated at 120 digits (tests/golden/closed_forms.txt), exact special
cases, invariants that hold for every input, library routines (scipy's
log_softmax and entropy), an exactly rounded pure-Python restatement, and
central finite differences of the forward for the gradient.  A dropped term, a
wrong sign, a wrong index or a transposed operand in the oracle fails at least
one of them (tests/test_oracle_mutations.py checks that claim).

Definitions: torchtitan PR #4685 "[RL] Avoid full-vocab gather for TP policy
statistics" (Summary, Why, Correctness and compatibility; logprob = -CE per
its review diff).
"""
import math
import os
import zlib

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle
from oracle import bruteforce, lmhead

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_forms.txt")
IGN = -100


def _golden():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, V, k, a, b, lpa, lpb, H = line.split()
            rows.append((name, int(V), int(k), float(a), float(b), float(lpa), float(lpb), float(H)))
    return rows


def _as(dtype, z64):
    if dtype == "f32":
        return z64.astype(np.float32)
    if dtype == "bf16":
        bits = oracle.bf16_bits(z64.astype(np.float32))
        assert np.array_equal(oracle.bf16_to_f64(bits), z64), "test values must be bf16-exact"
        return bits
    return z64


@pytest.mark.parametrize("dtype", ["f64", "f32", "bf16"])
@pytest.mark.parametrize("case", _golden(), ids=lambda c: c[0])
def test_closed_forms(case, dtype):
    name, V, k, a, b, lpa, lpb, H = case
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    row = np.full(V, b)
    pos = rng.permutation(V)[:k]
    row[pos] = a
    z = np.stack([row, row])
    ib = int(np.flatnonzero(row == b)[0]) if k < V else int(pos[0])
    labels = np.array([pos[0], ib], np.int64)
    out = oracle.forward(_as(dtype, z), labels, IGN)
    # left-to-right summation of V terms in double: relative error <= V * 2^-53
    rel = 2 * V * 2.0**-53 + 1e-13
    assert abs(out["logprob"][0] - lpa) <= rel * max(1.0, abs(lpa))
    assert abs(out["logprob"][1] - lpb) <= rel * max(1.0, abs(lpb))
    assert np.all(np.abs(out["entropy"] - H) <= rel * max(1.0, abs(H)))


def test_single_finite_entry():
    V = 1000
    z = np.full((3, V), -np.inf)
    z[:, 17] = 2.5
    out = oracle.forward(z, np.array([17, 3, IGN]), IGN)
    assert out["logprob"][0] == 0.0
    assert out["logprob"][1] == -np.inf
    assert out["logprob"][2] == 0.0
    assert np.all(out["entropy"] == 0.0)
    g = oracle.backward(z, np.array([17, 3, IGN]), np.array([1.5, 2.0, 3.0]), IGN)
    assert np.all(g[0] == 0.0)  # w (1 - 1) at the label, w (0 - 0) elsewhere
    assert g[1, 3] == 2.0 and g[1, 17] == -2.0 and np.count_nonzero(g[1]) == 2
    assert np.all(g[2] == 0.0)


def _rand_rows(rng, T, V, scale=3.0):
    return rng.standard_normal((T, V)) * scale


@pytest.mark.parametrize("V", [7, 1000, 4099])
def test_matches_scipy(V):
    rng = np.random.default_rng(V)
    z = _rand_rows(rng, 6, V)
    labels = rng.integers(0, V, 6)
    out = oracle.forward(z, labels, IGN)
    ls = scipy.special.log_softmax(z, axis=1)
    assert np.allclose(out["logprob"], ls[np.arange(6), labels], rtol=0, atol=1e-12)
    H = scipy.stats.entropy(np.exp(ls), axis=1)
    assert np.allclose(out["entropy"], H, rtol=1e-12, atol=1e-12)
    assert np.allclose(out["M"] + out["logS"], scipy.special.logsumexp(z, axis=1), rtol=0, atol=1e-12)


def test_bruteforce_tiny():
    """Tiny configuration (64 x 1000, N(0, 3^2), 5 ignored rows) against the
    exactly rounded pure-Python restatement."""
    rng = np.random.default_rng(0)
    T, V = 64, 1000
    z = (rng.standard_normal((T, V)) * 3.0).astype(np.float32)
    labels = rng.integers(0, V, T)
    labels[rng.permutation(T)[:5]] = IGN
    w = rng.standard_normal(T)
    out = oracle.forward(z, labels, IGN)
    g = oracle.backward(z, labels, w, IGN)
    for t in range(T):
        row = [float(x) for x in z[t]]
        lp, H = bruteforce.forward_row(row, int(labels[t]), IGN)
        assert abs(out["logprob"][t] - lp) <= 1e-13 * max(1, abs(lp))
        assert abs(out["entropy"][t] - H) <= 1e-13 * max(1, abs(H))
        if t < 8:
            gb = np.array(bruteforce.backward_row(row, int(labels[t]), float(w[t]), IGN))
            assert np.allclose(g[t], gb, rtol=1e-13, atol=1e-16)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_shift_invariance(dtype):
    """Adding a constant to every logit of a row changes nothing.  The grid is
    chosen so the shifted values stay exact in the input dtype."""
    rng = np.random.default_rng(5)
    T, V = 8, 1500
    if dtype == "f32":
        z = np.round(rng.uniform(-63, 63, (T, V)) * 1024) / 1024
        c = 37.0
    else:
        z = np.round(rng.uniform(-15.5, 15.5, (T, V)) * 4) / 4
        c = 32.0
    labels = rng.integers(0, V, T)
    w = rng.standard_normal(T)
    a = oracle.forward(_as(dtype, z), labels, IGN)
    b = oracle.forward(_as(dtype, z + c), labels, IGN)
    assert np.allclose(a["logprob"], b["logprob"], rtol=0, atol=1e-11)
    assert np.allclose(a["entropy"], b["entropy"], rtol=0, atol=1e-11)
    assert np.allclose(b["M"] - a["M"], c, rtol=0, atol=0)
    ga = oracle.backward(_as(dtype, z), labels, w, IGN)
    gb = oracle.backward(_as(dtype, z + c), labels, w, IGN)
    assert np.allclose(ga, gb, rtol=1e-11, atol=1e-15)


def test_gradient_sums_to_zero_and_scales_with_weight():
    rng = np.random.default_rng(6)
    T, V = 10, 2000
    z = _rand_rows(rng, T, V, 2.0)
    z[3, rng.permutation(V)[:200]] = -np.inf
    labels = rng.integers(0, V, T)
    labels[3] = int(np.flatnonzero(np.isfinite(z[3]))[0])
    labels[7] = IGN
    w = rng.standard_normal(T)
    g = oracle.backward(z, labels, w, IGN)
    sums = g.sum(axis=1)
    assert np.all(np.abs(sums) <= 1e-12 * np.maximum(np.abs(w), 1e-300))
    g1 = oracle.backward(z, labels, np.ones(T), IGN)
    assert np.allclose(g, g1 * w[:, None], rtol=1e-15, atol=0)
    # the label column holds w (1 - p_y) and every other column -w p_v
    p = np.exp(z - scipy.special.logsumexp(z, axis=1, keepdims=True))
    t = 0
    assert math.isclose(g[t, labels[t]], w[t] * (1 - p[t, labels[t]]), rel_tol=1e-13)
    other = (labels[t] + 1) % V
    assert math.isclose(g[t, other], -w[t] * p[t, other], rel_tol=1e-13)


def test_gradient_matches_finite_differences():
    """d logprob_y / d z_v = 1[v = y] - p_v, checked by central differences of
    the oracle's own forward (an independent path through the code)."""
    rng = np.random.default_rng(7)
    V = 40
    z = rng.standard_normal((1, V)) * 2.0
    y = 11
    g = oracle.backward(z, np.array([y]), np.array([1.0]), IGN)[0]
    h = 1e-6
    for v in range(V):
        zp, zm = z.copy(), z.copy()
        zp[0, v] += h
        zm[0, v] -= h
        fp = oracle.forward(zp, np.array([y]), IGN)["logprob"][0]
        fm = oracle.forward(zm, np.array([y]), IGN)["logprob"][0]
        fd = (fp - fm) / (2 * h)
        assert abs(fd - g[v]) <= 1e-7 * max(1.0, abs(g[v])), v


@pytest.mark.parametrize("bounds", [[0, 512, 1000], [0, 513, 1000], [0, 1, 999, 1000],
                                    [0, 250, 500, 750, 1000]])
def test_sharded_equals_full(bounds):
    rng = np.random.default_rng(8)
    T, V = 16, 1000
    z = _rand_rows(rng, T, V)
    z[2, bounds[0]:bounds[1]] = -np.inf      # a shard with no finite entry
    z[5, rng.permutation(V)[:100]] = -np.inf  # partially masked row
    labels = rng.integers(0, V, T)
    labels[2] = bounds[1]
    labels[5] = int(np.flatnonzero(np.isfinite(z[5]))[3])
    labels[9] = IGN
    full = oracle.forward(z, labels, IGN)
    sh = oracle.sharded(z, labels, bounds, IGN)
    assert np.allclose(sh["logprob"], full["logprob"], rtol=0, atol=1e-12)
    assert np.allclose(sh["entropy"], full["entropy"], rtol=0, atol=1e-12)
    # each shard's local values are those of the shard's columns alone
    s = 1
    sub = oracle.forward(z[:, bounds[s]:bounds[s + 1]], None, IGN)
    st = sh["shard_stats"][:, s]
    ok = np.isfinite(sub["M"])
    assert np.allclose(st[ok, 0], sub["M"][ok], rtol=0, atol=0)
    assert np.allclose(np.log(st[ok, 1]), sub["logS"][ok], rtol=0, atol=1e-12)


def test_permutation_invariance():
    rng = np.random.default_rng(9)
    T, V = 6, 3001
    z = _rand_rows(rng, T, V)
    labels = rng.integers(0, V, T)
    perm = rng.permutation(V)
    inv = np.argsort(perm)
    a = oracle.forward(z, labels, IGN)
    b = oracle.forward(z[:, perm], inv[labels], IGN)
    assert np.allclose(a["logprob"], b["logprob"], rtol=0, atol=1e-12)
    assert np.allclose(a["entropy"], b["entropy"], rtol=0, atol=1e-12)
    w = rng.standard_normal(T)
    ga = oracle.backward(z, labels, w, IGN)
    gb = oracle.backward(z[:, perm], inv[labels], w, IGN)
    assert np.allclose(ga[:, perm], gb, rtol=1e-12, atol=1e-18)


def test_ignored_and_masked():
    rng = np.random.default_rng(10)
    T, V = 5, 800
    z = _rand_rows(rng, T, V)
    mask = rng.permutation(V)[:80]
    z[1, mask] = -np.inf
    labels = np.array([IGN, 5, IGN, 7, 9])
    labels[1] = int(np.flatnonzero(np.isfinite(z[1]))[0])
    w = rng.standard_normal(T)
    w[3] = 0.0
    out = oracle.forward(z, labels, IGN)
    assert out["logprob"][0] == 0.0 and out["logprob"][2] == 0.0
    # entropy does not depend on the label: an ignored row still reports it
    ref = oracle.forward(z, np.array([1, 1, 1, 1, 1]), IGN)
    assert np.array_equal(out["entropy"], ref["entropy"])
    g = oracle.backward(z, labels, w, IGN)
    assert np.all(g[0] == 0) and np.all(g[2] == 0) and np.all(g[3] == 0)
    assert not np.any(np.signbit(g[0]))  # written as +0.0
    assert np.all(g[1, mask] == 0.0)
    # masking a column equals dropping it
    keep = np.setdiff1d(np.arange(V), mask)
    sub = oracle.forward(z[1:2, keep], np.array([int(np.searchsorted(keep, labels[1]))]), IGN)
    assert abs(sub["logprob"][0] - out["logprob"][1]) <= 1e-12
    assert abs(sub["entropy"][0] - out["entropy"][1]) <= 1e-12


def test_bad_labels_and_empty_rows_give_nan():
    z = np.zeros((3, 10))
    z[2] = -np.inf
    out = oracle.forward(z, np.array([10, -5, 0]), IGN)
    assert np.all(np.isnan(out["logprob"])) and np.all(np.isnan(out["entropy"]))


def test_lmhead_logits_match_bruteforce_dot():
    rng = np.random.default_rng(11)
    T, V, d = 4, 9, 33
    h = oracle.bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    W = oracle.bf16_bits((0.02 * rng.standard_normal((V, d))).astype(np.float32))
    z = lmhead.logits(h, W)
    hf, Wf = oracle.bf16_to_f64(h), oracle.bf16_to_f64(W)
    for t in range(T):
        for v in range(V):
            ref = math.fsum(float(hf[t, k]) * float(Wf[v, k]) for k in range(d))
            assert abs(z[t, v] - ref) <= 1e-15 * max(1e-3, abs(ref))


def test_lmhead_backward_matches_finite_differences():
    """dhidden and dW are the gradients of sum_t w_t logprob_t through z = h W^T."""
    rng = np.random.default_rng(12)
    T, V, d = 3, 11, 5
    h = rng.standard_normal((T, d))
    W = rng.standard_normal((V, d)) * 0.5
    labels = np.array([2, IGN, 7])
    w = np.array([0.7, 1.3, -1.1])
    dh, dW = lmhead.backward(h, W, labels, w, IGN)

    def f(hh, WW):
        lp = lmhead.forward(hh, WW, labels, IGN)["logprob"]
        return float(np.dot(w, lp))

    eps = 1e-6
    for t in range(T):
        for k in range(d):
            hp, hm = h.copy(), h.copy()
            hp[t, k] += eps
            hm[t, k] -= eps
            fd = (f(hp, W) - f(hm, W)) / (2 * eps)
            assert abs(fd - dh[t, k]) <= 1e-7 * max(1.0, abs(dh[t, k]))
    for v in range(V):
        for k in range(d):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, k] += eps
            Wm[v, k] -= eps
            fd = (f(h, Wp) - f(h, Wm)) / (2 * eps)
            assert abs(fd - dW[v, k]) <= 1e-7 * max(1.0, abs(dW[v, k]))


# ---- loss-side epilogue (oracle/policy.py) ----------------------------------
from oracle import policy as opol  # noqa: E402


def test_diff_metrics_hand_example():
    pi = np.array([1.0, 2.0, 3.0, 4.0], np.float32)
    mu = np.array([1.0, 1.5, 5.0, 9.0], np.float32)
    lab = np.array([0, 1, 2, IGN])          # the last token is ignored
    m = opol.diff_metrics(pi, mu, lab, IGN)  # d = (0, 0.5, -2)
    assert m["mean"] == -0.5 and m["abs_mean"] == 2.5 / 3 and m["max"] == 2.0
    assert m["different"] == 2 / 3


def test_diff_metrics_bitwise_and_degenerate():
    z = np.array([0.0], np.float32)
    nz = np.array([-0.0], np.float32)
    m = opol.diff_metrics(z, nz, [0], IGN)   # equal values, different bits
    assert m["mean"] == 0.0 and m["abs_mean"] == 0.0 and m["different"] == 1.0
    same = opol.diff_metrics(np.arange(5, dtype=np.float32), np.arange(5, dtype=np.float32),
                             np.arange(5), IGN)
    assert same == {"mean": 0.0, "abs_mean": 0.0, "max": 0.0, "different": 0.0}
    none = opol.diff_metrics(np.ones(3, np.float32), np.zeros(3, np.float32), [IGN] * 3, IGN)
    assert math.isnan(none["mean"]) and none["max"] == 0.0 and math.isnan(none["different"])


@pytest.mark.parametrize("adv,lr,loss,weight", [
    (1.0, 0.0, -1.0, -1.0),                               # r = 1: unclipped
    (1.0, 0.5, -1.28, 0.0),                               # r > 1.28, A > 0: clipped, no gradient
    (-1.0, 0.5, math.exp(0.5), math.exp(0.5)),            # r > 1.28, A < 0: unclipped
    (1.0, -0.5, -math.exp(-0.5), -math.exp(-0.5)),        # r < 0.8, A > 0: unclipped
    (-1.0, -0.5, 0.8, 0.0),                               # r < 0.8, A < 0: clipped
    (2.0, 0.1, -2.0 * math.exp(0.1), -2.0 * math.exp(0.1)),
])
def test_clipped_surrogate_cases(adv, lr, loss, weight):
    l, w = opol.clipped_surrogate([lr], [0.0], [adv], [0], 0.2, 0.28, 1.0, IGN)
    assert math.isclose(l[0], loss, rel_tol=1e-15, abs_tol=1e-15)
    assert math.isclose(w[0], weight, rel_tol=1e-15, abs_tol=1e-15)
    l2, w2 = opol.clipped_surrogate([lr], [0.0], [adv], [IGN], 0.2, 0.28, 1.0, IGN)
    assert l2[0] == 0.0 and w2[0] == 0.0
    l3, w3 = opol.clipped_surrogate([lr], [0.0], [adv], [0], 0.2, 0.28, 0.25, IGN)
    assert math.isclose(l3[0], 0.25 * loss, abs_tol=1e-15) and math.isclose(w3[0], 0.25 * weight, abs_tol=1e-15)


def test_clipped_surrogate_weight_is_the_derivative():
    rng = np.random.default_rng(13)
    old = rng.normal(-3, 1, 200)
    pi = old + rng.normal(0, 0.3, 200)
    adv = rng.normal(0, 1, 200)
    lab = np.zeros(200, np.int64)
    _, w = opol.clipped_surrogate(pi, old, adv, lab)
    h = 1e-6
    lp, _ = opol.clipped_surrogate(pi + h, old, adv, lab)
    lm, _ = opol.clipped_surrogate(pi - h, old, adv, lab)
    fd = (lp - lm) / (2 * h)
    r = np.exp(pi - old)
    away = (np.abs(r - 0.8) > 1e-4) & (np.abs(r - 1.28) > 1e-4)  # not at a kink
    assert np.allclose(fd[away], w[away], rtol=1e-6, atol=1e-9)


def test_log_softmax_matches_scipy_and_normalises():
    rng = np.random.default_rng(21)
    z = rng.standard_normal((5, 3001)) * 3
    z[2, :100] = -np.inf
    ls = oracle.log_softmax(z)
    ref = scipy.special.log_softmax(z, axis=1)
    fin = np.isfinite(ref)
    assert np.allclose(ls[fin], ref[fin], rtol=0, atol=1e-12)
    assert np.all(np.isneginf(ls[~fin]))
    assert np.allclose(np.exp(ls).sum(axis=1), 1.0, rtol=0, atol=1e-12)
