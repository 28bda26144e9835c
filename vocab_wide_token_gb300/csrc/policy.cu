// policy.cu -- the loss side of the policy statistics.
//
// pstat_logprob_diff_metrics: the trainer/rollout mismatch metrics that the
//   torchtitan batch-invariant GDN README logs (bit_wise/logprob_diff/{mean,
//   abs_mean, max} and bit_wise/ratio_tokens_different/mean), computed on the
//   device in one fixed-order reduction, so the same inputs give the same
//   bits every time.
// pstat_clipped_surrogate: the clipped-ratio surrogate of that README's DAPO
//   recipes (clip (0.2, 0.28)), per token, and its derivative with respect to
//   the logprob -- the per-token weight that pstat_backward /
//   pstat_forward_backward multiply (onehot - softmax) by.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"

namespace pstat {
namespace {

constexpr int kMetricThreads = 1024;

// One CTA: thread i takes tokens i, i + 1024, ... in order (double-precision
// sums), then a fixed shared-memory tree combines the threads.
__global__ void __launch_bounds__(kMetricThreads)
    diff_metrics_kernel(const float* __restrict__ pi, const float* __restrict__ mu,
                        const int64_t* __restrict__ labels, int64_t ignore_index, int64_t T,
                        float* __restrict__ out) {
    __shared__ double s_sum[kMetricThreads], s_abs[kMetricThreads];
    __shared__ double s_max[kMetricThreads];
    __shared__ long long s_n[kMetricThreads], s_diff[kMetricThreads];
    const int i = threadIdx.x;
    double sum = 0.0, sabs = 0.0;
    double mx = 0.0;
    long long n = 0, ndiff = 0;
    for (int64_t t = i; t < T; t += kMetricThreads) {
        if (labels && labels[t] == ignore_index) continue;
        const float a = pi[t], b = mu[t];
        const double d = (double)a - (double)b;  // exact
        sum += d;
        sabs += fabs(d);
        mx = fmax(mx, fabs(d));
        ++n;
        ndiff += (__float_as_uint(a) != __float_as_uint(b));
    }
    s_sum[i] = sum;
    s_abs[i] = sabs;
    s_max[i] = mx;
    s_n[i] = n;
    s_diff[i] = ndiff;
    __syncthreads();
    for (int stride = kMetricThreads / 2; stride > 0; stride >>= 1) {
        if (i < stride) {
            s_sum[i] += s_sum[i + stride];
            s_abs[i] += s_abs[i + stride];
            s_max[i] = fmax(s_max[i], s_max[i + stride]);
            s_n[i] += s_n[i + stride];
            s_diff[i] += s_diff[i + stride];
        }
        __syncthreads();
    }
    if (i == 0) {
        const long long cnt = s_n[0];
        out[0] = cnt ? (float)(s_sum[0] / (double)cnt) : NAN;
        out[1] = cnt ? (float)(s_abs[0] / (double)cnt) : NAN;
        out[2] = (float)s_max[0];
        out[3] = cnt ? (float)((double)s_diff[0] / (double)cnt) : NAN;
    }
}

// r = e^(pi - pi_old); loss = -scale min(r A, clip(r, 1 - eps_low, 1 + eps_high) A);
// weight = dloss/dpi = -scale A r when the unclipped term is the minimum (or
// ties), else 0.  Ignored tokens: loss 0, weight 0.
__global__ void __launch_bounds__(256)
    clipped_surrogate_kernel(const float* __restrict__ pi, const float* __restrict__ pi_old,
                             const float* __restrict__ adv, const int64_t* __restrict__ labels,
                             int64_t ignore_index, int64_t T, float eps_low, float eps_high,
                             float scale, float* __restrict__ loss, float* __restrict__ weight) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    float l = 0.f, w = 0.f;
    if (!labels || labels[t] != ignore_index) {
        const float a = adv[t];
        const float r = expf(pi[t] - pi_old[t]);
        const float rc = fminf(fmaxf(r, 1.f - eps_low), 1.f + eps_high);
        const float unclipped = r * a, clipped = rc * a;
        if (unclipped <= clipped) {
            l = -scale * unclipped;
            w = -scale * a * r;
        } else {
            l = -scale * clipped;
        }
    }
    if (loss) loss[t] = l;
    weight[t] = w;
}

}  // namespace
}  // namespace pstat

using namespace pstat;

extern "C" int pstat_logprob_diff_metrics(const float* logprob, const float* rollout_logprob,
                                          const int64_t* labels, int64_t ignore_index, int64_t T,
                                          float* out_metrics, pstat_stream_t stream) {
    if (T < 0) return PSTAT_ERR_SHAPE;
    if (!out_metrics || (T > 0 && (!logprob || !rollout_logprob))) return PSTAT_ERR_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(logprob) & 3u) || (reinterpret_cast<uintptr_t>(rollout_logprob) & 3u) ||
        (reinterpret_cast<uintptr_t>(out_metrics) & 3u) ||
        (labels && (reinterpret_cast<uintptr_t>(labels) & 7u)))
        return PSTAT_ERR_ALIGN;
    DeviceInfo dev;
    const int rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    diff_metrics_kernel<<<1, kMetricThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        logprob, rollout_logprob, labels, ignore_index, T, out_metrics);
    return cudaGetLastError() == cudaSuccess ? PSTAT_OK : PSTAT_ERR_CUDA;
}

extern "C" int pstat_clipped_surrogate(const float* logprob, const float* old_logprob,
                                       const float* advantages, const int64_t* labels,
                                       int64_t ignore_index, int64_t T, float eps_low,
                                       float eps_high, float scale, float* out_loss,
                                       float* out_weight, pstat_stream_t stream) {
    if (T < 0 || !(eps_low >= 0.f) || !(eps_high >= 0.f) || !(eps_low < 1.f)) return PSTAT_ERR_SHAPE;
    if (T == 0) return PSTAT_OK;
    if (!logprob || !old_logprob || !advantages || !out_weight) return PSTAT_ERR_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(logprob) & 3u) || (reinterpret_cast<uintptr_t>(old_logprob) & 3u) ||
        (reinterpret_cast<uintptr_t>(advantages) & 3u) || (reinterpret_cast<uintptr_t>(out_weight) & 3u) ||
        (out_loss && (reinterpret_cast<uintptr_t>(out_loss) & 3u)) ||
        (labels && (reinterpret_cast<uintptr_t>(labels) & 7u)))
        return PSTAT_ERR_ALIGN;
    DeviceInfo dev;
    const int rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    const unsigned grid = (unsigned)((T + 255) / 256);
    clipped_surrogate_kernel<<<grid, 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        logprob, old_logprob, advantages, labels, ignore_index, T, eps_low, eps_high, scale,
        out_loss, out_weight);
    return cudaGetLastError() == cudaSuccess ? PSTAT_OK : PSTAT_ERR_CUDA;
}
