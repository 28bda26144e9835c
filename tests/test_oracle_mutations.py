"""Plants plausible mistakes in copies of the oracle's C source and checks that
the pins in test_oracle_pins.py catch every one of them.

Each mutant is compiled with gcc into a temporary directory and loaded through
ORACLE_LIB by a child pytest run of the pin suite; the mutation test passes
only when that child run fails.  Nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "pstat_oracle.c")

# (id, original text, mutated text): each original must occur exactly once.
MUTANTS = [
    ("entropy_sign", "H -= p * (x - L);", "H += p * (x - L);"),
    ("entropy_dropped_shift", "H -= p * (x - L);", "H -= p * x;"),
    ("label_off_by_one", "lp = load_elem(z, dtype, ld, t, y) - L;",
     "lp = load_elem(z, dtype, ld, t, (y + 1) % V) - L;"),
    ("denominator_skips_first", "if (x > -INFINITY) S += exp(x - M);",
     "if (x > -INFINITY && v > 0) S += exp(x - M);"),
    ("grad_sign", "row[v] = w * (onehot - p);", "row[v] = w * (p - onehot);"),
    ("grad_no_onehot", "row[v] = w * (onehot - p);", "row[v] = -w * p;"),
    ("grad_unweighted", "row[v] = w * (onehot - p);", "row[v] = (onehot - p);"),
    ("logS_output", "if (logS_out) logS_out[t] = (M > -INFINITY) ? log(S) : NAN;",
     "if (logS_out) logS_out[t] = (M > -INFINITY) ? log(S) + 1e-9 : NAN;"),
    ("shard_no_rescale", "S += ms[3 * s + 1] * r;", "S += ms[3 * s + 1];"),
    ("shard_u_dropped_term", "U += r * (ms[3 * s + 2] + (m - M) * ms[3 * s + 1]);",
     "U += r * ms[3 * s + 2];"),
    ("shard_bounds_transposed", "for (int64_t v = bounds[s]; v < bounds[s + 1]; ++v) {\n                double x = load_elem(z, dtype, ld, t, v);\n                if (x > m) m = x;",
     "for (int64_t v = bounds[s]; v < bounds[s + 1]; ++v) {\n                double x = load_elem(z, dtype, ld, v % T, t % V);\n                if (x > m) m = x;"),
    ("bf16_wrong_shift", "uint32_t bits = ((uint32_t)((const uint16_t*)z)[idx]) << 16;",
     "uint32_t bits = ((uint32_t)((const uint16_t*)z)[idx]) << 15;"),
]


@pytest.mark.parametrize("mid,orig,mut", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(mid, orig, mut, tmp_path):
    src = open(SRC).read()
    assert src.count(orig) == 1, f"mutation anchor for {mid} not unique"
    mpath = tmp_path / "mutant.c"
    mpath.write_text(src.replace(orig, mut))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(lib),
                    str(mpath), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {mid} survived the pins:\n{r.stdout[-2000:]}"
