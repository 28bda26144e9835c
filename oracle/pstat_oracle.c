/*
 * pstat_oracle.c -- float64 CPU oracle for per-token policy statistics.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA path is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product library never links, calls or falls back to it.  It shares no
 * source, header, table or helper with the CUDA code.
 *
 * What it computes (torchtitan PR #4685, "[RL] Avoid full-vocab gather for
 * TP policy statistics": Summary, Why, and the review diff that defines
 * logprobs as the negated cross entropy):
 *   for every token row t with logits z_t[0..V):
 *     M_t   = max_v z_tv                                  (global maximum)
 *     S_t   = sum_v exp(z_tv - M_t)                        (softmax denominator)
 *     L_t   = M_t + ln S_t                                 (log partition)
 *     logprob_t = z_{t,y_t} - L_t     (0 when y_t is the ignore index)
 *     entropy_t = -sum_{v: z_tv > -inf} p_tv (z_tv - L_t),  p_tv = exp(z_tv - L_t)
 *     dlogits_tv = w_t (1[v = y_t] - p_tv)   (an all-zero row when ignored)
 * The gradient is that of the per-token cross entropy (same page, "reuse
 * vocab-parallel cross-entropy forward/backward for per-token gradients"),
 * scaled by the per-token weight w_t ("non-uniformly weighted gradients",
 * Correctness and compatibility).
 *
 * Every sum runs left to right over ascending v in double precision; no
 * blocking, chunking or reordering.  The only parallelism is OpenMP over
 * independent rows.
 *
 * The sharded routine (oracle_sharded) restates, also in double precision,
 * the reduction the page describes for tensor-parallel shards: each shard
 * holds a local maximum, a local sum of exponentials and a local
 * entropy-weighted sum; a MAX reduction and SUM reductions combine them
 * (torchtitan PR #4685, "[RL] Avoid full-vocab gather for TP policy
 * statistics", the review thread on batch invariance: each shard sums the
 * exponentials of its logits shifted by the global maximum, then a SUM
 * all-reduce adds the shards).
 * It exists to check the invariant "shard-combined statistics equal the
 * full-vocabulary statistics".
 *
 * Input element types: 0 = float32, 1 = bfloat16 (raw 16-bit patterns),
 * 2 = float64.  Conversion of float32 and bfloat16 to double is exact.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F32 0
#define ORACLE_BF16 1
#define ORACLE_F64 2

static int g_threads = 0; /* 0: OpenMP default */

void oracle_set_threads(int n) { g_threads = n; }

int oracle_threads(void) {
#ifdef _OPENMP
    return g_threads > 0 ? g_threads : omp_get_max_threads();
#else
    return 1;
#endif
}

/* Element v of row t, widened to double.  bfloat16 is the upper half of a
 * float32, so shifting its 16 bits up by 16 gives the float32 with the same
 * value. */
static double load_elem(const void* z, int dtype, int64_t ld, int64_t t, int64_t v) {
    int64_t idx = t * ld + v;
    if (dtype == ORACLE_F32) {
        return (double)((const float*)z)[idx];
    } else if (dtype == ORACLE_BF16) {
        uint32_t bits = ((uint32_t)((const uint16_t*)z)[idx]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return ((const double*)z)[idx];
}

static int bad_args(const void* z, int dtype, int64_t T, int64_t V, int64_t ld) {
    if (T < 0 || V < 1 || ld < V) return 1;
    if (T > 0 && z == NULL) return 1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64) return 1;
    return 0;
}

/* Row statistics by the plain definition: two passes over the full row. */
static void row_stats(const void* z, int dtype, int64_t ld, int64_t t, int64_t V,
                      double* M_out, double* S_out) {
    double M = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double x = load_elem(z, dtype, ld, t, v);
        if (x > M) M = x;
    }
    double S = 0.0;
    if (M > -INFINITY) {
        for (int64_t v = 0; v < V; ++v) {
            double x = load_elem(z, dtype, ld, t, v);
            if (x > -INFINITY) S += exp(x - M);
        }
    }
    *M_out = M;
    *S_out = S;
}

/*
 * Forward: logprob and entropy per row, plus (M, ln S) per row.
 * Any of the outputs may be NULL.  A label outside [0, V) that is not the
 * ignore index gives NaN outputs for that row.  A row with no finite entry
 * has an undefined softmax and gives NaN outputs.
 * Returns 0, or -1 on bad arguments.
 */
int oracle_forward(const void* z, int dtype, int64_t T, int64_t V, int64_t ld,
                   const int64_t* labels, int64_t ignore_index,
                   double* logprob, double* entropy, double* M_out, double* logS_out) {
    if (bad_args(z, dtype, T, V, ld)) return -1;
    int nt = oracle_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t t = 0; t < T; ++t) {
        double M, S;
        row_stats(z, dtype, ld, t, V, &M, &S);
        double lp, H;
        if (!(M > -INFINITY)) {
            lp = NAN;
            H = NAN;
        } else {
            double L = M + log(S);
            H = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                double x = load_elem(z, dtype, ld, t, v);
                if (x > -INFINITY) {
                    double p = exp(x - L);
                    H -= p * (x - L);
                }
            }
            int64_t y = labels ? labels[t] : ignore_index;
            if (y == ignore_index) {
                lp = 0.0;
            } else if (y < 0 || y >= V) {
                lp = NAN;
                H = NAN;
            } else {
                lp = load_elem(z, dtype, ld, t, y) - L;
            }
        }
        if (logprob) logprob[t] = lp;
        if (entropy) entropy[t] = H;
        if (M_out) M_out[t] = M;
        if (logS_out) logS_out[t] = (M > -INFINITY) ? log(S) : NAN;
    }
    return 0;
}

/*
 * Backward: dlogits[t, v] = w_t (1[v = y_t] - p_tv), written densely into
 * out[t * V + v] (row stride V).  Rows whose label is the ignore index, or
 * whose weight is exactly zero, are all +0.0.  weights may be NULL (all 1).
 */
int oracle_backward(const void* z, int dtype, int64_t T, int64_t V, int64_t ld,
                    const int64_t* labels, int64_t ignore_index, const double* weights,
                    double* out) {
    if (bad_args(z, dtype, T, V, ld) || (T > 0 && out == NULL)) return -1;
    int nt = oracle_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t t = 0; t < T; ++t) {
        double* row = out + t * V;
        int64_t y = labels ? labels[t] : ignore_index;
        double w = weights ? weights[t] : 1.0;
        if (y == ignore_index || w == 0.0) {
            for (int64_t v = 0; v < V; ++v) row[v] = 0.0;
            continue;
        }
        double M, S;
        row_stats(z, dtype, ld, t, V, &M, &S);
        if (!(M > -INFINITY) || y < 0 || y >= V) {
            for (int64_t v = 0; v < V; ++v) row[v] = NAN;
            continue;
        }
        double L = M + log(S);
        for (int64_t v = 0; v < V; ++v) {
            double x = load_elem(z, dtype, ld, t, v);
            double p = (x > -INFINITY) ? exp(x - L) : 0.0;
            double onehot = (v == y) ? 1.0 : 0.0;
            row[v] = w * (onehot - p);
        }
    }
    return 0;
}

/*
 * Sharded statistics in double precision.  bounds[0..n_shards] must be
 * strictly increasing from 0 to V.  For every row and shard s the shard-local
 * values over columns [bounds[s], bounds[s+1]) are
 *   m_s = max z,  s_s = sum exp(z - m_s),  u_s = sum exp(z - m_s) (z - m_s)
 * written to shard_stats[(t * n_shards + s) * 3 + {0,1,2}] when non-NULL.
 * The row is then combined: M = max_s m_s, and every shard's sums are moved
 * to the common maximum,
 *   S = sum_s s_s exp(m_s - M),
 *   U = sum_s exp(m_s - M) (u_s + (m_s - M) s_s),
 * giving logprob = z_y - M - ln S and entropy = ln S - U / S.
 * Shards with no finite entry (m_s = -inf) contribute nothing.
 */
int oracle_sharded(const void* z, int dtype, int64_t T, int64_t V, int64_t ld,
                   const int64_t* labels, int64_t ignore_index,
                   const int64_t* bounds, int n_shards,
                   double* shard_stats, double* logprob, double* entropy) {
    if (bad_args(z, dtype, T, V, ld) || n_shards < 1 || bounds == NULL) return -1;
    if (bounds[0] != 0 || bounds[n_shards] != V) return -1;
    for (int s = 0; s < n_shards; ++s)
        if (bounds[s + 1] <= bounds[s]) return -1;
    int nt = oracle_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int64_t t = 0; t < T; ++t) {
        double M = -INFINITY;
        double* ms = (double*)malloc(sizeof(double) * 3 * (size_t)n_shards);
        for (int s = 0; s < n_shards; ++s) {
            double m = -INFINITY;
            for (int64_t v = bounds[s]; v < bounds[s + 1]; ++v) {
                double x = load_elem(z, dtype, ld, t, v);
                if (x > m) m = x;
            }
            double ss = 0.0, uu = 0.0;
            if (m > -INFINITY) {
                for (int64_t v = bounds[s]; v < bounds[s + 1]; ++v) {
                    double x = load_elem(z, dtype, ld, t, v);
                    if (x > -INFINITY) {
                        double e = exp(x - m);
                        ss += e;
                        uu += e * (x - m);
                    }
                }
            }
            ms[3 * s + 0] = m;
            ms[3 * s + 1] = ss;
            ms[3 * s + 2] = uu;
            if (shard_stats) {
                shard_stats[(t * n_shards + s) * 3 + 0] = m;
                shard_stats[(t * n_shards + s) * 3 + 1] = ss;
                shard_stats[(t * n_shards + s) * 3 + 2] = uu;
            }
            if (m > M) M = m;
        }
        double S = 0.0, U = 0.0;
        if (M > -INFINITY) {
            for (int s = 0; s < n_shards; ++s) {
                double m = ms[3 * s + 0];
                if (!(m > -INFINITY)) continue;
                double r = exp(m - M);
                S += ms[3 * s + 1] * r;
                U += r * (ms[3 * s + 2] + (m - M) * ms[3 * s + 1]);
            }
        }
        free(ms);
        double lp, H;
        if (!(M > -INFINITY)) {
            lp = NAN;
            H = NAN;
        } else {
            double lnS = log(S);
            H = lnS - U / S;
            int64_t y = labels ? labels[t] : ignore_index;
            if (y == ignore_index) {
                lp = 0.0;
            } else if (y < 0 || y >= V) {
                lp = NAN;
                H = NAN;
            } else {
                lp = load_elem(z, dtype, ld, t, y) - M - lnS;
            }
        }
        if (logprob) logprob[t] = lp;
        if (entropy) entropy[t] = H;
    }
    return 0;
}
