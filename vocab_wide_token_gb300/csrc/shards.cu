// shards.cu -- vocabulary-parallel use: each rank holds the logits of one
// vocabulary shard [b_s, b_{s+1}) of every row.
//
//   pstat_shard_stats     per row, the shard's statistics (M_s, S_s, U_s, z_y):
//                         chunks laid from the shard start and folded in the
//                         fixed order, by the forward kernel;
//   pstat_combine_shards  the fixed-order combine of the gathered [T, S, 4]
//                         statistics (shards in ascending vocabulary order)
//                         into logprob, entropy and (M, ln S);
//   pstat_backward_shard  the weighted backward of the shard's columns from
//                         the global (M, ln S).
//
// The exchange between ranks is an all-gather of the [T, 4] statistics (not
// a sum), after which every rank runs the same combine on the same bits.
// The in-shard fold and the cross-shard step are the two levels of the
// sharded forward's fold, so shard_stats on every shard followed by
// combine_shards gives bit for bit what pstat_forward gives with those
// shard_bounds, and backward_shard gives that shard's columns of
// pstat_backward.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "chunk_math.cuh"
#include "internal.h"

namespace pstat {
namespace {

struct ShardStarts {
    int64_t b[PSTAT_MAX_SHARDS + 1];
    int n;
};

// One thread per row: shards in ascending order, as in the sharded fold.
__global__ void __launch_bounds__(256)
    combine_shards_kernel(const float4* __restrict__ st, const __grid_constant__ ShardStarts sb,
                          int64_t T, const int64_t* __restrict__ labels, int64_t ignore_index,
                          float* __restrict__ logprob, float* __restrict__ entropy,
                          float* __restrict__ rowstats, int* __restrict__ dev_error) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int n = sb.n;
    const float4* r = st + t * n;
    float M = -INFINITY;
    for (int s = 0; s < n; ++s) M = fmaxf(M, r[s].x);
    float S = 0.f, U = 0.f;
    if (M > -INFINITY) {
        for (int s = 0; s < n; ++s) {
            const float4 q = r[s];
            if (q.x == -INFINITY) continue;  // fully masked shard
            fold_shard(q.x, q.y, q.z, M, S, U);
        }
    }
    const int64_t V = sb.b[n];
    int err = 0;
    float lnS, H, lp;
    if (!(M > -INFINITY)) {
        err |= PSTAT_DEV_EMPTY_ROW;
        lnS = NAN;
        H = NAN;
        lp = NAN;
    } else {
        lnS = logf(S);
        H = lnS - U / S;
        const int64_t y = labels ? labels[t] : ignore_index;
        if (y == ignore_index) {
            lp = 0.f;
        } else if (y < 0 || y >= V) {
            err |= PSTAT_DEV_BAD_LABEL;
            lp = NAN;
            H = NAN;
        } else {
            int s = 0;
            while (sb.b[s + 1] <= y) ++s;  // the shard that holds column y
            lp = (r[s].w - M) - lnS;
        }
    }
    if (logprob) logprob[t] = lp;
    if (entropy) entropy[t] = H;
    if (rowstats) reinterpret_cast<float2*>(rowstats)[t] = make_float2(M, lnS);
    if (err && dev_error) atomicOr(dev_error, err);
}

bool valid_dtype(int dt) { return dt == PSTAT_F32 || dt == PSTAT_BF16; }
size_t elem_size(pstat_dtype dt) { return dt == PSTAT_BF16 ? 2 : 4; }
bool misaligned(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a); }

}  // namespace
}  // namespace pstat

using namespace pstat;

extern "C" int pstat_shard_stats(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                 int64_t ld, const int64_t* labels, int64_t ignore_index,
                                 int64_t vocab_start, float* out_stats, int* dev_error,
                                 pstat_stream_t stream) {
    if (!valid_dtype(dt)) return PSTAT_ERR_DTYPE;
    if (T < 0 || V < 1 || ld < V || vocab_start < 0) return PSTAT_ERR_SHAPE;
    ShardPlan plan;
    int rc = make_plan(V, dt == PSTAT_BF16 ? PSTAT_CHUNK_BF16 : PSTAT_CHUNK_F32, nullptr, 1, &plan);
    if (rc != PSTAT_OK) return rc;
    if (plan.n_chunks > forward_rows_max_chunks()) return PSTAT_ERR_SHAPE;
    if (T == 0) return PSTAT_OK;
    if (!logits || !out_stats) return PSTAT_ERR_NULLPTR;
    if (misaligned(logits, elem_size(dt)) || misaligned(out_stats, 16) || misaligned(labels, 8))
        return PSTAT_ERR_ALIGN;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    return launch_forward_rows(logits, dt, T, V, ld, plan, labels, ignore_index, nullptr, nullptr,
                               nullptr, dev_error, dev, reinterpret_cast<cudaStream_t>(stream),
                               reinterpret_cast<float4*>(out_stats), vocab_start) == cudaSuccess
               ? PSTAT_OK
               : PSTAT_ERR_CUDA;
}

extern "C" int pstat_combine_shards(const float* stats, int64_t T, int n_shards,
                                    const int64_t* shard_bounds, const int64_t* labels,
                                    int64_t ignore_index, float* out_logprob, float* out_entropy,
                                    float* out_rowstats, int* dev_error, pstat_stream_t stream) {
    if (T < 0) return PSTAT_ERR_SHAPE;
    if (!shard_bounds || n_shards < 1 || n_shards > PSTAT_MAX_SHARDS) return PSTAT_ERR_SHARDS;
    ShardStarts sb;
    sb.n = n_shards;
    for (int s = 0; s <= n_shards; ++s) {
        sb.b[s] = shard_bounds[s];
        if ((s == 0 && sb.b[0] != 0) || (s > 0 && sb.b[s] <= sb.b[s - 1])) return PSTAT_ERR_SHARDS;
    }
    if (T == 0) return PSTAT_OK;
    if (!stats) return PSTAT_ERR_NULLPTR;
    if (misaligned(stats, 16) || misaligned(labels, 8) || misaligned(out_rowstats, 8) ||
        misaligned(out_logprob, 4) || misaligned(out_entropy, 4))
        return PSTAT_ERR_ALIGN;
    DeviceInfo dev;
    const int rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    const unsigned grid = (unsigned)((T + 255) / 256);
    combine_shards_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        reinterpret_cast<const float4*>(stats), sb, T, labels, ignore_index, out_logprob,
        out_entropy, out_rowstats, dev_error);
    return cudaGetLastError() == cudaSuccess ? PSTAT_OK : PSTAT_ERR_CUDA;
}

extern "C" int pstat_backward_shard(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                    int64_t ld, const int64_t* labels, int64_t ignore_index,
                                    const float* weights, const float* rowstats,
                                    int64_t vocab_start, int64_t vocab_total, void* out_dlogits,
                                    pstat_dtype out_dt, int64_t ld_out, int* dev_error,
                                    pstat_stream_t stream) {
    if (!valid_dtype(dt) || !valid_dtype(out_dt)) return PSTAT_ERR_DTYPE;
    if (dt == PSTAT_BF16 && out_dt == PSTAT_F32) return PSTAT_ERR_DTYPE;
    if (T < 0 || V < 1 || ld < V || ld_out < V || vocab_start < 0 || vocab_start + V > vocab_total)
        return PSTAT_ERR_SHAPE;
    if (T == 0) return PSTAT_OK;
    if (!logits || !out_dlogits || !rowstats) return PSTAT_ERR_NULLPTR;
    if (misaligned(logits, elem_size(dt)) || misaligned(out_dlogits, elem_size(out_dt)) ||
        misaligned(rowstats, 8) || misaligned(labels, 8) || misaligned(weights, 4))
        return PSTAT_ERR_ALIGN;
    DeviceInfo dev;
    const int rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    return launch_backward(logits, dt, T, V, ld, labels, ignore_index, weights, rowstats,
                           out_dlogits, out_dt, ld_out, dev_error, dev,
                           reinterpret_cast<cudaStream_t>(stream), vocab_start,
                           vocab_total) == cudaSuccess
               ? PSTAT_OK
               : PSTAT_ERR_CUDA;
}
