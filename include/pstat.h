/*
 * pstat.h -- C ABI of libpstat.so: batch-invariant per-token policy
 * statistics over a wide vocabulary on one GB300 (sm_103a).
 *
 * What the library computes is defined in torchtitan PR #4685, "[RL] Avoid
 * full-vocab gather for TP policy statistics":
 *   - Summary / Why: per-token sampled-token logprob and exact entropy from
 *     shard-local sufficient statistics (global maximum, softmax
 *     denominator, target contribution, entropy-weighted sum); entropy is a
 *     no-grad metric.
 *   - Review diff of loss.py: logprobs = -cross_entropy(logits, labels).
 *   - Correctness and compatibility: even/uneven vocabulary shards, FP32 and
 *     BF16 logits, ignored labels, partially masked (-inf) logits, and
 *     non-uniformly weighted gradients compared with the full vocabulary.
 * The fused lm_head entry points follow the chunked lm_head of TRL PR #6949
 * "ZeroSyncGRPOTrainer" (the vocabulary projection is multiplied chunk by
 * chunk; backward GEMMs run in bf16 and accumulate in fp32).
 *
 * Per row t with logits z_t[0..V), label y_t and weight w_t:
 *   M_t       = max_v z_tv,   S_t = sum_v exp(z_tv - M_t)
 *   logprob_t = z_{t,y_t} - M_t - ln S_t          (+0.0 if y_t == ignore_index)
 *   entropy_t = ln S_t - U_t / S_t,  U_t = sum_v exp(z_tv - M_t)(z_tv - M_t)
 *               (computed for ignored rows too: it does not depend on y_t)
 *   dlogits_tv = w_t (1[v = y_t] - exp(z_tv - M_t - ln S_t))
 *               (an all +0.0 row when y_t == ignore_index or w_t == 0)
 *
 * Numerics and batch invariance.  Each row is cut into fixed chunks that
 * restart at every shard start: chunk k of shard s covers columns
 * [b_s + k C, min(b_s + (k+1) C, b_{s+1})), C = PSTAT_CHUNK_BF16 or
 * PSTAT_CHUNK_F32 elements.  Per chunk the kernel forms (m, s, u) with a
 * reduction tree fixed at compile time; within a shard the chunks are folded
 * by a fixed tree (32 lane-strided ascending partial sums, then an xor
 * butterfly) and shards in ascending order within the row.  A row's
 * results therefore depend only on its own values, V, the shard bounds and
 * the dtype: they are bit-identical whatever batch the row sits in, at
 * whatever position, and from call to call.  Sharded and unsharded results
 * agree to rounding, not bitwise (the page's point that a partial sum then a
 * SUM reduction differs in the low bits from one contiguous sum).
 *
 * Conventions for every entry point:
 *   - All pointers except `shard_bounds` are DEVICE pointers owned by the
 *     caller (typically torch tensors).  `shard_bounds` is a HOST array.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The library allocates no memory; scratch lives in the
 *     caller's `workspace`, sized by the matching *_workspace_size call.
 *   - Errors a host can see (null pointers, shapes, shard bounds, dtype,
 *     alignment, workspace size) are returned before anything is launched.
 *     A launch failure returns PSTAT_ERR_CUDA (from cudaGetLastError).
 *   - Errors only the device can see are OR-ed into `*dev_error` (a device
 *     int, may be NULL) with atomics, and the affected row's outputs become
 *     NaN; no kernel traps or asserts.  Read the flag when you need it.
 *   - Labels are int64, weights float32, statistics and logprob/entropy
 *     float32.  Logits/dlogits are row-major with a row stride `ld` (in
 *     elements, >= V).
 */
#ifndef PSTAT_H
#define PSTAT_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PSTAT_API __attribute__((visibility("default")))
#else
#define PSTAT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle; identical to cudaStream_t. */
typedef struct CUstream_st* pstat_stream_t;

typedef enum { PSTAT_F32 = 0, PSTAT_BF16 = 1 } pstat_dtype;

/* Return codes. */
enum {
    PSTAT_OK = 0,
    PSTAT_ERR_NULLPTR = -1,     /* a required pointer is NULL */
    PSTAT_ERR_SHAPE = -2,       /* T < 0, V < 1, ld < V, d not a multiple of 64, ... */
    PSTAT_ERR_SHARDS = -3,      /* bounds not strictly increasing from 0 to V, or too many */
    PSTAT_ERR_DTYPE = -4,       /* unknown dtype or unsupported combination */
    PSTAT_ERR_ALIGN = -5,       /* a pointer lacks the alignment stated for it */
    PSTAT_ERR_WORKSPACE = -6,   /* workspace NULL or smaller than required */
    PSTAT_ERR_CUDA = -7,        /* a CUDA runtime call or launch failed */
    PSTAT_ERR_UNSUPPORTED = -8  /* the current device is not sm_103 (GB300) */
};

/* Bits OR-ed into *dev_error by the kernels. */
#define PSTAT_DEV_BAD_LABEL 0x1 /* label outside [0, V) and != ignore_index */
#define PSTAT_DEV_EMPTY_ROW 0x2 /* every logit of a row is -inf: softmax undefined */
#define PSTAT_DEV_TIMEOUT 0x4   /* a bounded wait on an asynchronous copy gave up */
#define PSTAT_DEV_RANGE 0x8     /* lm_head backward: a value exceeds the fp16 range (65504) */

#define PSTAT_MAX_SHARDS 64
#define PSTAT_CHUNK_BF16 4096 /* chunk length in elements for bf16 logits */
#define PSTAT_CHUNK_F32 2048  /* chunk length in elements for fp32 logits */

/* Human-readable text for a return code; never NULL. */
PSTAT_API const char* pstat_status_string(int code);

/* Version of this ABI (major * 10000 + minor * 100 + patch). */
PSTAT_API int pstat_version(void);

/*
 * Workspace bytes for pstat_forward / pstat_backward on T rows of V logits
 * of dtype `dt` split by `shard_bounds` (host, n_shards + 1 entries; NULL and
 * n_shards = 1 mean one shard {0, V}).  The workspace holds one 16-byte
 * (m, s, u) record per row and chunk, and the (M, ln S) pair per row that
 * pstat_backward needs when it is not given `rowstats`.
 */
PSTAT_API int pstat_workspace_size(int64_t T, int64_t V, pstat_dtype dt, const int64_t* shard_bounds,
                         int n_shards, size_t* bytes);

/*
 * Forward statistics: per-chunk statistics combined in a fixed order.  Plans
 * of at most 256 chunks per row run as one kernel with the records in shared
 * memory (no workspace needed: it may be NULL and is not touched); larger
 * plans run the chunk-statistics kernel into the workspace, then the combine.
 * Both give the same bits.
 *   logits        [T, ld] dtype `dt`; element (t, v) at logits + t*ld + v.
 *                 Any alignment works; 16-byte aligned rows and chunk starts
 *                 take the bulk-copy path, others a slower path with the same
 *                 numerics.
 *   labels        [T] int64 (NULL: every row ignored).
 *   shard_bounds  host int64[n_shards + 1], 0 = b_0 < b_1 < ... < b_S = V,
 *                 n_shards <= PSTAT_MAX_SHARDS; NULL means {0, V}.
 *   out_logprob   [T] float (may be NULL), out_entropy [T] float (may be
 *                 NULL), out_rowstats [T, 2] float (M, ln S) (may be NULL).
 *   workspace     >= pstat_workspace_size(...) bytes, 16-byte aligned;
 *                 required only for plans of more than 256 chunks per row
 *                 (PSTAT_ERR_WORKSPACE when it is missing there).
 *   dev_error     device int or NULL; bits PSTAT_DEV_*.
 * T = 0 is a no-op returning PSTAT_OK.
 */
PSTAT_API int pstat_forward(const void* logits, pstat_dtype dt, int64_t T, int64_t V, int64_t ld,
                  const int64_t* labels, int64_t ignore_index, const int64_t* shard_bounds,
                  int n_shards, float* out_logprob, float* out_entropy, float* out_rowstats,
                  void* workspace, size_t ws_bytes, int* dev_error, pstat_stream_t stream);

/* Bytes of the fixed device scratch used by pstat_forward_noalloc (8 MiB). */
#define PSTAT_NOALLOC_SCRATCH_BYTES (8u << 20)

/* PSTAT_NOALLOC_SCRATCH_BYTES as built into this library, for bindings that
 * cannot read the header. */
PSTAT_API size_t pstat_noalloc_scratch_bytes(void);

/*
 * pstat_forward for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for this library's
 * users.  Some callers must not call cudaMalloc where they compute these
 * statistics: allocation synchronises the device, a host runtime or
 * framework may own all device memory through its own pool, or a plain C
 * caller may have no allocator at all.  This variant takes no workspace and
 * allocates nothing: its per-chunk scratch is a fixed array of
 * PSTAT_NOALLOC_SCRATCH_BYTES inside the library, present on every GPU that
 * loads the library until the process exits.  The caller still passes the
 * inputs and outputs, with the same meaning, layout and results as
 * pstat_forward.
 *   Limit: T * n_chunks * 16 bytes must fit the scratch (n_chunks as in
 *   pstat_workspace_size; e.g. T <= 13,797 rows at V = 151,936 in bf16),
 *   else PSTAT_ERR_WORKSPACE is returned before anything is launched.
 *   The first call on each device looks up the scratch's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.  The address is cached per CUDA context
 *   (cuCtxGetId): after cudaDeviceReset, the first call in the new context
 *   looks it up again, so that call too belongs before any capture.
 *   Every call on a device shares the one scratch array, which keeps the last
 *   call's contents.  Nothing in it needs clearing (each call writes every
 *   record it reads), but calls whose kernels overlap on the GPU (different
 *   streams, or host threads issuing concurrently) race on it: serialise
 *   them, e.g. on one stream.
 */
PSTAT_API int pstat_forward_noalloc(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                    int64_t ld, const int64_t* labels, int64_t ignore_index,
                                    const int64_t* shard_bounds, int n_shards, float* out_logprob,
                                    float* out_entropy, float* out_rowstats, int* dev_error,
                                    pstat_stream_t stream);

/*
 * Weighted backward dlogits = w (onehot(y) - softmax(z)) (fused elementwise
 * kernel).
 *   weights       [T] float (NULL: all ones).
 *   rowstats      [T, 2] float (M, ln S) from pstat_forward on the same
 *                 logits and shard bounds; NULL recomputes them first through
 *                 the forward kernels (needs the workspace).
 *   out_dlogits   [T, ld_out] of `out_dt` (PSTAT_BF16 rounds to nearest even;
 *                 PSTAT_F32 needs dt == PSTAT_F32).  Every element of the
 *                 T x V block is written.
 *   workspace     needed only when rowstats is NULL (else may be NULL / 0).
 */
PSTAT_API int pstat_backward(const void* logits, pstat_dtype dt, int64_t T, int64_t V, int64_t ld,
                   const int64_t* labels, int64_t ignore_index, const float* weights,
                   const float* rowstats, const int64_t* shard_bounds, int n_shards,
                   void* out_dlogits, pstat_dtype out_dt, int64_t ld_out, void* workspace,
                   size_t ws_bytes, int* dev_error, pstat_stream_t stream);

/*
 * pstat_forward followed by pstat_backward in one pass over the logits
 * (the pages' forward+backward unit, reusing cross-entropy forward and
 * backward together; here as one kernel).  Results are bit-identical to the
 * two calls with the same arguments; the logits are read from HBM once (each
 * CTA re-reads a row's chunks from L2 for the gradient), so a bf16 token
 * moves 4V bytes instead of 6V.  No workspace: a row's chunk records live in
 * shared memory.
 *   Arguments as in pstat_forward / pstat_backward; out_dlogits [T, ld_out]
 *   is required, out_logprob / out_entropy / out_rowstats may be NULL.
 *   The shard plan may have at most 256 chunks per row (PSTAT_ERR_SHAPE).
 */
PSTAT_API int pstat_forward_backward(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                     int64_t ld, const int64_t* labels, int64_t ignore_index,
                                     const float* weights, const int64_t* shard_bounds,
                                     int n_shards, float* out_logprob, float* out_entropy,
                                     float* out_rowstats, void* out_dlogits, pstat_dtype out_dt,
                                     int64_t ld_out, int* dev_error, pstat_stream_t stream);

/*
 * Vocabulary-parallel use: each rank holds the logits of one vocabulary shard
 * [b_s, b_{s+1}) of every row (torchtitan PR #4685, Summary and the review
 * thread's batch-invariance answer: shard-local maximum, sum of exponentials,
 * entropy-weighted sum and target logit, reduced across ranks).  Here the
 * ranks exchange the [T, 4] statistics with an all-gather instead of MAX/SUM
 * all-reduces, and every rank folds them in ascending shard order with
 * pstat_combine_shards, so all ranks hold the same bits and the result does
 * not depend on the collective's reduction order.
 *
 * pstat_shard_stats on every shard followed by pstat_combine_shards equals
 * pstat_forward with those shard_bounds bit for bit; pstat_backward_shard
 * equals the shard's columns of pstat_backward.
 */

/*
 * Per-row statistics of one vocabulary shard.
 *   logits        [T, ld] dtype `dt`: this shard's V columns (chunks are laid
 *                 from its first column).  V may hold at most 256 chunks
 *                 (PSTAT_ERR_SHAPE otherwise).
 *   labels        [T] int64 in the whole vocabulary's numbering, or NULL.
 *   vocab_start   the shard's first column in that numbering (b_s).
 *   out_stats     [T, 4] float, 16-byte aligned: (M_s, S_s, U_s, z_y) with
 *                 S_s = sum exp(z - M_s), U_s = sum exp(z - M_s)(z - M_s) over
 *                 the shard, and z_y the label's logit when vocab_start <= y <
 *                 vocab_start + V, else 0.  A fully masked shard gives
 *                 (-inf, 0, 0, .).  Label range errors are reported by
 *                 pstat_combine_shards.
 */
PSTAT_API int pstat_shard_stats(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                int64_t ld, const int64_t* labels, int64_t ignore_index,
                                int64_t vocab_start, float* out_stats, int* dev_error,
                                pstat_stream_t stream);

/*
 * Fixed-order combine of gathered shard statistics into the row outputs.
 *   stats         [T, n_shards, 4] float (device, 16-byte aligned): row t,
 *                 shard s at stats + (t n_shards + s) 4, shards in ascending
 *                 vocabulary order.
 *   shard_bounds  host int64[n_shards + 1], 0 = b_0 < ... < b_S = V_total.
 *   Outputs, labels and dev_error as pstat_forward (bad labels: bit 1, NaN;
 *   fully masked rows: bit 2, NaN).
 */
PSTAT_API int pstat_combine_shards(const float* stats, int64_t T, int n_shards,
                                   const int64_t* shard_bounds, const int64_t* labels,
                                   int64_t ignore_index, float* out_logprob, float* out_entropy,
                                   float* out_rowstats, int* dev_error, pstat_stream_t stream);

/*
 * Weighted backward of one vocabulary shard's columns.
 *   As pstat_backward on the shard's V columns, with rowstats [T, 2] the
 *   global (M, ln S) (required) and labels in the whole vocabulary's
 *   numbering: the one-hot term lands in this shard only when vocab_start <=
 *   y < vocab_start + V; labels outside [0, vocab_total) give NaN rows and
 *   dev_error bit 1.  vocab_start + V <= vocab_total.
 */
PSTAT_API int pstat_backward_shard(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                   int64_t ld, const int64_t* labels, int64_t ignore_index,
                                   const float* weights, const float* rowstats,
                                   int64_t vocab_start, int64_t vocab_total, void* out_dlogits,
                                   pstat_dtype out_dt, int64_t ld_out, int* dev_error,
                                   pstat_stream_t stream);

/*
 * The full log-softmax log p_tv = z_tv - M_t - ln S_t as a [T, V] tensor, in
 * one read and one write pass over the logits, from the same row statistics
 * as the other entry points (so it is batch-invariant too: a row's output
 * bits do not depend on the batch).  The BI log_softmax of the batch-
 * invariant GDN README's kernel list, for callers that need every column.
 *   rowstats  [T, 2] (M, ln S) from pstat_forward with the same shard bounds,
 *             or NULL to compute them first (needs the workspace).
 *   out       [T, ld_out] of out_dt (bf16 rounds to nearest even); -inf
 *             logits give -inf, rows with no finite logit give NaN and set
 *             PSTAT_DEV_EMPTY_ROW.
 */
PSTAT_API int pstat_log_softmax(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                int64_t ld, const float* rowstats, const int64_t* shard_bounds,
                                int n_shards, void* out, pstat_dtype out_dt, int64_t ld_out,
                                void* workspace, size_t ws_bytes, int* dev_error,
                                pstat_stream_t stream);

/*
 * Trainer/rollout logprob mismatch metrics, as the torchtitan batch-invariant
 * GDN README logs them ("Code map": bit_wise/logprob_diff/{mean,abs_mean,max}
 * and bit_wise/ratio_tokens_different/mean).  Over the tokens whose label is
 * not ignore_index (all tokens when labels is NULL), d_t = logprob_t -
 * rollout_logprob_t:
 *   out_metrics[0] = mean d,  [1] = mean |d|,  [2] = max |d|,
 *   [3] = fraction of tokens whose float32 bit patterns differ.
 * With no token counted: [0], [1], [3] are NaN and [2] is 0.  One fixed-order
 * reduction on the device (double-precision sums): repeated calls give the
 * same bits.  logprob, rollout_logprob [T] float; out_metrics device float[4].
 */
PSTAT_API int pstat_logprob_diff_metrics(const float* logprob, const float* rollout_logprob,
                                         const int64_t* labels, int64_t ignore_index, int64_t T,
                                         float* out_metrics, pstat_stream_t stream);

/*
 * Clipped-ratio policy surrogate (the DAPO recipes of the same README use
 * eps_low = 0.2, eps_high = 0.28), per token, with r_t = exp(logprob_t -
 * old_logprob_t):
 *   out_loss_t   = -scale min(r_t A_t, clip(r_t, 1 - eps_low, 1 + eps_high) A_t)
 *   out_weight_t = d out_loss_t / d logprob_t
 *                = -scale A_t r_t if the unclipped term is the minimum (or
 *                  ties), else 0 (the clipped term does not depend on logprob).
 * Ignored tokens get loss 0 and weight 0.  out_weight is what pstat_backward
 * and pstat_forward_backward take as `weights` to give the loss's gradient
 * with respect to the logits.  All arrays [T] float (out_loss may be NULL);
 * 0 <= eps_low < 1, eps_high >= 0.
 */
PSTAT_API int pstat_clipped_surrogate(const float* logprob, const float* old_logprob,
                                      const float* advantages, const int64_t* labels,
                                      int64_t ignore_index, int64_t T, float eps_low,
                                      float eps_high, float scale, float* out_loss,
                                      float* out_weight, pstat_stream_t stream);

/*
 * Workspace bytes for the fused lm_head entry points (T tokens, V vocab
 * rows, hidden size d).
 */
PSTAT_API int pstat_lmhead_workspace_size(int64_t T, int64_t V, int64_t d, size_t* bytes);

/*
 * Fused lm_head forward: logits z = hidden W^T are formed tile by tile on
 * the tensor cores (bf16 operands, fp32 accumulation in tensor memory) and
 * folded straight into the chunk statistics; logits are never written to
 * memory.  Outputs as pstat_forward.
 *   hidden  [T, d] bf16 row-major, W [V, d] bf16 row-major; both 16-byte
 *           aligned, d a multiple of 64 (PSTAT_ERR_SHAPE otherwise).
 */
PSTAT_API int pstat_lmhead_fused(const void* hidden, const void* W, int64_t T, int64_t V, int64_t d,
                       const int64_t* labels, int64_t ignore_index, float* out_logprob,
                       float* out_entropy, float* out_rowstats, void* workspace,
                       size_t ws_bytes, int* dev_error, pstat_stream_t stream);

/*
 * Fused lm_head backward through z = hidden W^T of the weighted gradient
 * g = w (onehot(y) - softmax(z)):
 *   dhidden [T, d] float  += g W
 *   dW      [V, d] float  += g^T hidden
 * Both are ACCUMULATED into (zero them first for a plain gradient), so calls
 * over token or vocabulary chunks compose.  rowstats [T, 2] from
 * pstat_lmhead_fused is required.  g is formed on chip from recomputed
 * logits and staged only per vocabulary chunk in the workspace.
 */
PSTAT_API int pstat_lmhead_backward(const void* hidden, const void* W, int64_t T, int64_t V, int64_t d,
                          const int64_t* labels, int64_t ignore_index, const float* weights,
                          const float* rowstats, float* dhidden, float* dW, void* workspace,
                          size_t ws_bytes, int* dev_error, pstat_stream_t stream);

/*
 * Self-test of the bounded waits.  Every kernel of this library waits on its
 * mbarriers for at most a fixed time (2 s); a wait that runs out sets
 * PSTAT_DEV_TIMEOUT in *dev_error and the kernel winds down instead of
 * hanging the GPU.  This entry point runs one such wait, limited to
 * `limit_ns` nanoseconds (at most 1e9, else PSTAT_ERR_SHAPE), on a barrier
 * that nothing arrives at, with no copy in flight: afterwards *dev_error
 * (a device int, required) has PSTAT_DEV_TIMEOUT set and the context is
 * usable as before.  The pages have no counterpart; it exists to test the
 * library's failure path without faulting or hanging a GPU.
 */
PSTAT_API int pstat_selftest_wait_timeout(uint64_t limit_ns, int* dev_error,
                                          pstat_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PSTAT_H */
