// stats_kernels.cu -- the memory-bound hot path on sm_103a.
//
//  K-A chunk_stats_kernel : per (row, chunk) sufficient statistics
//                           m = max z, s = sum e^(z-m), u = sum e^(z-m)(z-m)
//  K-B combine_kernel     : fixed-order fold of the chunk statistics into
//                           per-shard, then per-row (M, S, U); writes logprob,
//                           entropy and (M, ln S)
//  K-C backward_kernel    : dlogits = w (onehot(y) - e^(z - M - ln S))
//
// The statistics are those of torchtitan PR #4685 ("[RL] Avoid full-vocab
// gather for TP policy statistics", Why): global maximum, softmax
// denominator, target contribution and entropy-weighted sum.  The page
// reduces them across tensor-parallel ranks with a MAX then SUM all-reduces;
// here the same algebra folds fixed chunks in a fixed order on one GPU, which
// is what makes every row's result independent of the batch around it.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "chunk_math.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace pstat {

// ---------------------------------------------------------------------------
// K-A: chunk statistics.
//
// Persistent CTAs of kWarps warps, one CTA per SM.  The flattened list of
// (row, chunk) items is split into one contiguous range per warp.  Every warp
// owns a ring of kStages shared-memory slots of 8 KB; its lane 0 streams
// chunks into the ring with 1-D bulk asynchronous copies (the TMA engine)
// that complete on one mbarrier per slot.  A chunk is read out of its slot
// once, into registers (lane L holds the 16-byte vectors L, L+32, ..., L+480:
// 64 registers), and the slot is refilled at once with the chunk kStages
// ahead, so copies stay in flight while the warp computes.
// Chunks whose start or byte length is not 16-byte aligned cannot use the
// bulk copy; the warp loads those element by element into the same slot
// (padded with -inf to whole vectors).  The reduction sees the same values in
// the same registers either way, so the numerics do not depend on alignment
// or on which warp processes the chunk.
//
// The per-chunk arithmetic is described in chunk_math.cuh.
// ---------------------------------------------------------------------------
template <typename E>
__global__ void __launch_bounds__(kWarps * 32, 1)
    chunk_stats_kernel(const E* __restrict__ logits, int64_t T, int64_t ld,
                       const __grid_constant__ ShardPlan plan, float4* __restrict__ out,
                       int* __restrict__ dev_error) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* slots = smem + (size_t)warp * kStages * kSlotBytes;
    uint64_t* bars =
        reinterpret_cast<uint64_t*>(smem + (size_t)kWarps * kStages * kSlotBytes) + warp * kStages;

    const int64_t n_items = T * plan.n_chunks;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp;
    const int64_t nw = (int64_t)gridDim.x * kWarps;
    const int64_t i0 = n_items * gw / nw;
    const int64_t i1 = n_items * (gw + 1) / nw;
    const int64_t n = i1 - i0;
    if (n <= 0) return;

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    const uint64_t policy = policy_evict_first();

    // Item i is chunk g of row t with i = t n_chunks + g; both the consuming
    // and the issuing position walk the items in order, so (t, g) is advanced
    // instead of divided out per item.
    struct Item {
        int64_t t;
        int g;
    };
    auto next_item = [&](Item& it) {
        if (++it.g == plan.n_chunks) {
            it.g = 0;
            ++it.t;
        }
    };
    auto locate = [&](const Item& it, const E*& src, int& len) -> bool {
        int64_t start;
        chunk_span(plan, it.g, start, len);
        src = logits + it.t * ld + start;
        return ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) &&
               ((((size_t)len * sizeof(E)) & 15u) == 0);
    };
    auto issue = [&](const Item& it, int slot) {
        const E* src;
        int len;
        if (locate(it, src, len) && lane == 0) {
            const uint32_t bytes = (uint32_t)len * (uint32_t)sizeof(E);
            mbar_arrive_expect_tx(&bars[slot], bytes);
            bulk_g2s_hint(slots + (size_t)slot * kSlotBytes, src, bytes, &bars[slot], policy);
        }
    };

    Item cur = {i0 / plan.n_chunks, (int)(i0 % plan.n_chunks)};
    Item ahead = cur;
    const int64_t prologue = n < kStages ? n : kStages;
    for (int64_t j = 0; j < prologue; ++j) {
        issue(ahead, (int)j);
        next_item(ahead);
    }

    uint32_t phase = 0;  // parity bit per slot, flipped after each bulk completion
    int64_t j = 0;
    bool timed_out = false;
    for (; j < n; ++j) {
        const int slot = (int)(j % kStages);
        E* buf = reinterpret_cast<E*>(slots + (size_t)slot * kSlotBytes);
        const E* src;
        int len;
        if (locate(cur, src, len)) {
            bool ok = mbar_wait_bounded(&bars[slot], (phase >> slot) & 1u, kWaitLimitNs);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) {
                timed_out = true;
                break;
            }
            phase ^= 1u << slot;
        } else {
            // Unaligned chunk: element loads, padded with -inf to a whole vector.
            constexpr int kVec = Elem<E>::kVec;
            const int padded = (len + kVec - 1) / kVec * kVec;
            for (int k = lane; k < padded; k += 32) buf[k] = (k < len) ? src[k] : Elem<E>::neg_inf();
            __syncwarp();
        }
        uint4 q[kVecPerLane];
        load_chunk_regs<E>(buf, len, lane, q);
        __syncwarp();
        fence_proxy_async_smem();  // our reads of the slot precede the next bulk write into it
        if (j + kStages < n) {
            issue(ahead, slot);
            next_item(ahead);
        }
        const float4 r = reduce_regs(q, (E*)nullptr, len);
        if (lane == 0) out[i0 + j] = r;
        next_item(cur);
    }
    if (timed_out) {
        if (lane == 0 && dev_error) atomicOr(dev_error, PSTAT_DEV_TIMEOUT);
        // Drain copies still in flight into this CTA's shared memory before leaving.
        const int64_t last = (j + kStages < n) ? j + kStages : n;
        for (int64_t k = j; k < last; ++k) {
            const int slot = (int)(k % kStages);
            const E* src;
            int len;
            if (locate(cur, src, len)) {
                mbar_wait_bounded(&bars[slot], (phase >> slot) & 1u, kWaitLimitNs);
                phase ^= 1u << slot;
            }
            next_item(cur);
        }
    }
}

// ---------------------------------------------------------------------------
// K-B: fixed-order combine, one warp per row (fold_row_warp), then logprob,
// entropy and (M, ln S) from (M, S, U).
// ---------------------------------------------------------------------------
constexpr int kCombineWarps = 8;  // rows per CTA

template <typename E>
__global__ void __launch_bounds__(kCombineWarps * 32)
    combine_kernel(const float4* __restrict__ cs, const __grid_constant__ ShardPlan plan,
                   const E* __restrict__ logits, int64_t T, int64_t V, int64_t ld,
                   const int64_t* __restrict__ labels, int64_t ignore_index,
                   const float* __restrict__ target, float* __restrict__ logprob,
                   float* __restrict__ entropy, float* __restrict__ rowstats,
                   int* __restrict__ dev_error) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const float3 st = fold_row_warp(cs + t * plan.n_chunks, plan, lane);
    if (lane != 0) return;
    const float M = st.x, S = st.y, U = st.z;
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
            // target logit: from the logits, or recorded by the fused lm_head
            const float zy = target ? target[t] : Elem<E>::to_float(logits[t * ld + y]);
            lp = (zy - M) - lnS;
        }
    }
    if (logprob) logprob[t] = lp;
    if (entropy) entropy[t] = H;
    if (rowstats) reinterpret_cast<float2*>(rowstats)[t] = make_float2(M, lnS);
    if (err && dev_error) atomicOr(dev_error, err);
}

// ---------------------------------------------------------------------------
// K-C: weighted backward, elementwise.  Grid = T rows x `segs` column
// segments; each CTA streams its segment with 16-byte vector loads and
// stores (8 elements per step).  Rows that are ignored or carry a zero
// weight are written as +0.0 without reading the logits.
// ---------------------------------------------------------------------------
// An 8-element group loaded as raw 16-byte vectors (one for bf16, two for
// fp32) -> floats.
template <typename E>
__device__ __forceinline__ void unpack_group(const uint4 (&v)[(int)sizeof(E) / 2], float (&x)[8]);
template <>
__device__ __forceinline__ void unpack_group<uint16_t>(const uint4 (&v)[1], float (&x)[8]) {
    const uint32_t w[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        x[2 * e] = bf2_lo(w[e]);
        x[2 * e + 1] = bf2_hi(w[e]);
    }
}
template <>
__device__ __forceinline__ void unpack_group<float>(const uint4 (&v)[2], float (&x)[8]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        x[4 * h] = __uint_as_float(v[h].x);
        x[4 * h + 1] = __uint_as_float(v[h].y);
        x[4 * h + 2] = __uint_as_float(v[h].z);
        x[4 * h + 3] = __uint_as_float(v[h].w);
    }
}

constexpr int kBwdThreads = 256;
constexpr int kBwdUnroll = 4;

template <typename Ein, typename Eout>
__global__ void __launch_bounds__(kBwdThreads)
    backward_kernel(const Ein* __restrict__ logits, int64_t V, int64_t ld,
                    const int64_t* __restrict__ labels, int64_t ignore_index,
                    const float* __restrict__ weights, const float2* __restrict__ rowstats,
                    Eout* __restrict__ out, int64_t ld_out, int segs, int64_t label_offset,
                    int64_t v_total, int* __restrict__ dev_error) {
    // The columns are [label_offset, label_offset + V) of a vocabulary of
    // v_total (the whole row: 0 and V); labels are checked against v_total.
    const int64_t t = blockIdx.x / segs;
    const int seg = (int)(blockIdx.x - t * segs);
    const int64_t nv_row = V >> 3;  // whole 8-element groups in the row
    const int64_t c0 = (nv_row * seg / segs) << 3;
    const int64_t c1 = (seg == segs - 1) ? V : ((nv_row * (seg + 1) / segs) << 3);
    const Ein* zin = logits + t * ld;
    Eout* zout = out + t * ld_out;

    const int64_t y = labels ? labels[t] : ignore_index;
    const int64_t yl = y - label_offset;  // the label's column in this block of columns
    const float w = weights ? weights[t] : 1.f;
    int mode;  // 0: zero row, 1: NaN row, 2: compute
    GradRow row = {0.f, 0.f, 0.f, 0.f};
    if (y == ignore_index || w == 0.f) {
        mode = 0;
    } else {
        const float2 rs = rowstats[t];
        if (y < 0 || y >= v_total || !(rs.x > -INFINITY) || !(rs.y == rs.y)) {
            mode = 1;
            if (seg == 0 && threadIdx.x == 0 && dev_error)
                atomicOr(dev_error,
                         (y < 0 || y >= v_total) ? PSTAT_DEV_BAD_LABEL : PSTAT_DEV_EMPTY_ROW);
        } else {
            mode = 2;
            row = grad_row(rs.x, rs.y, w);
        }
    }
    const float fill = (mode == 0) ? 0.f : NAN;
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(zin + c0) & 15u) == 0) &&
                        ((reinterpret_cast<uintptr_t>(zout + c0) & 15u) == 0);
    const int64_t nv = vec_ok ? (c1 - c0) >> 3 : 0;

    // 8-element groups in flight per thread as raw 16-byte vectors, as in the
    // log-softmax kernel below: 6 bf16 groups (61 registers) took 0.643
    // against 0.650 ms for 4 unpacked ones and 0.652 for 8 raw ones (66
    // registers, one CTA fewer per SM) at T = 8192; fp32 1.328 against 1.360.
    constexpr int kVecs = (int)sizeof(Ein) / 2;
    constexpr int kU = kVecs == 1 ? 6 : kBwdUnroll;
    for (int64_t base = 0; base < nv; base += (int64_t)kBwdThreads * kU) {
        uint4 raw[kU][kVecs];
        int64_t col[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) {
            const int64_t i = base + (int64_t)k * kBwdThreads + threadIdx.x;
            col[k] = (i < nv) ? c0 + (i << 3) : -1;
            if (mode == 2 && col[k] >= 0) {
                const uint4* src = reinterpret_cast<const uint4*>(zin + col[k]);
#pragma unroll
                for (int h = 0; h < kVecs; ++h) raw[k][h] = __ldcs(src + h);
            }
        }
#pragma unroll
        for (int k = 0; k < kU; ++k) {
            if (col[k] < 0) continue;
            float g[8];
            if (mode == 2) {
                float x[8], ex[8];
                unpack_group<Ein>(raw[k], x);
                exp8(x, row.m2, ex);
                grad8(ex, row, g);
                const int64_t r = yl - col[k];
                if (r >= 0 && r < 8) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (e == r) g[e] = grad_label(ex[e], row);  // w (1 - p_y)
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) g[e] = fill;
            }
            Store8<Eout>::run(zout + col[k], g);
        }
    }
    // Scalar remainder: the tail of the segment, or all of it when unaligned.
    for (int64_t c = c0 + (nv << 3) + threadIdx.x; c < c1; c += kBwdThreads) {
        float g;
        if (mode == 2) {
            const float x = Elem<Ein>::to_float(zin[c]);
            const float e = ex2_approx(fmaf(x, kLog2e, -row.m2));
            g = (c == yl) ? grad_label(e, row) : e * row.nwK;
        } else {
            g = fill;
        }
        zout[c] = out_cast(g, zout);
    }
}

// ---------------------------------------------------------------------------
// Full log-softmax from the row statistics: out = (z - M) - ln S, element-
// wise, in the layout and with the streaming scheme of the backward kernel.
// Rows whose statistics are undefined (every logit -inf) are written as NaN.
// ---------------------------------------------------------------------------
template <typename Ein, typename Eout>
__global__ void __launch_bounds__(kBwdThreads)
    logsoftmax_kernel(const Ein* __restrict__ logits, int64_t V, int64_t ld,
                      const float2* __restrict__ rowstats, Eout* __restrict__ out, int64_t ld_out,
                      int segs, int* __restrict__ dev_error) {
    const int64_t t = blockIdx.x / segs;
    const int seg = (int)(blockIdx.x - t * segs);
    const int64_t nv_row = V >> 3;
    const int64_t c0 = (nv_row * seg / segs) << 3;
    const int64_t c1 = (seg == segs - 1) ? V : ((nv_row * (seg + 1) / segs) << 3);
    const Ein* zin = logits + t * ld;
    Eout* zout = out + t * ld_out;
    const float2 rs = rowstats[t];
    const bool defined = (rs.x > -INFINITY) && (rs.y == rs.y);
    if (!defined && seg == 0 && threadIdx.x == 0 && dev_error) atomicOr(dev_error, PSTAT_DEV_EMPTY_ROW);
    const float M = defined ? rs.x : NAN, lnS = defined ? rs.y : NAN;
    const uint64_t negM = f2_pack(-M, -M), nlnS = f2_pack(-lnS, -lnS);
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(zin + c0) & 15u) == 0) &&
                        ((reinterpret_cast<uintptr_t>(zout + c0) & 15u) == 0);
    const int64_t nv = vec_ok ? (c1 - c0) >> 3 : 0;
    // Each thread keeps kLsUnroll 8-element groups in flight as raw 16-byte
    // vectors (4 registers per bf16 group, not the 8 of unpacked floats): 8
    // bf16 groups at 48 registers gave 0.710 against 0.787 ms for 4 unpacked
    // groups at 60 registers (T = 8192, V = 151,936), the difference being
    // the bytes each SM keeps in flight.
    constexpr int kVecs = (int)sizeof(Ein) / 2;  // 16-byte vectors per group
    constexpr int kLsUnroll = kVecs == 1 ? 8 : kBwdUnroll;
    for (int64_t base = 0; base < nv; base += (int64_t)kBwdThreads * kLsUnroll) {
        uint4 raw[kLsUnroll][kVecs];
#pragma unroll
        for (int k = 0; k < kLsUnroll; ++k) {
            const int64_t i = base + (int64_t)k * kBwdThreads + threadIdx.x;
            if (i < nv) {
                const uint4* src = reinterpret_cast<const uint4*>(zin + c0 + (i << 3));
#pragma unroll
                for (int h = 0; h < kVecs; ++h) raw[k][h] = __ldcs(src + h);
            }
        }
#pragma unroll
        for (int k = 0; k < kLsUnroll; ++k) {
            const int64_t i = base + (int64_t)k * kBwdThreads + threadIdx.x;
            if (i >= nv) continue;
            float x[8];
            unpack_group<Ein>(raw[k], x);
            float o[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const uint64_t d = f2_add(f2_pack(x[2 * e], x[2 * e + 1]), negM);
                f2_unpack(f2_add(d, nlnS), o[2 * e], o[2 * e + 1]);
            }
            Store8<Eout>::run(zout + c0 + (i << 3), o);
        }
    }
    for (int64_t c = c0 + (nv << 3) + threadIdx.x; c < c1; c += kBwdThreads)
        zout[c] = out_cast((Elem<Ein>::to_float(zin[c]) - M) - lnS, zout);
}

// ---------------------------------------------------------------------------
// Launchers.
// ---------------------------------------------------------------------------
template <typename E>
static cudaError_t launch_chunk_stats_t(const E* logits, int64_t T, int64_t ld,
                                        const ShardPlan& plan, float4* cs, int* dev_error,
                                        const DeviceInfo& dev, cudaStream_t stream) {
    static ContextSeen configured;
    const size_t smem = chunk_stats_smem_bytes();
    const cudaError_t e = ensure_smem_optin(reinterpret_cast<const void*>(chunk_stats_kernel<E>),
                                            (int)smem, configured);
    if (e != cudaSuccess) return e;
    const int64_t items = T * plan.n_chunks;
    int64_t grid = (items + kWarps - 1) / kWarps;
    if (grid > dev.sm_count) grid = dev.sm_count;
    if (grid < 1) grid = 1;
    chunk_stats_kernel<E><<<(unsigned)grid, kWarps * 32, smem, stream>>>(logits, T, ld, plan, cs,
                                                                          dev_error);
    return cudaGetLastError();
}

cudaError_t launch_chunk_stats(const void* logits, pstat_dtype dt, int64_t T, int64_t ld,
                               const ShardPlan& plan, float4* cs, int* dev_error,
                               const DeviceInfo& dev, cudaStream_t stream) {
    if (dt == PSTAT_BF16)
        return launch_chunk_stats_t(static_cast<const uint16_t*>(logits), T, ld, plan, cs,
                                    dev_error, dev, stream);
    return launch_chunk_stats_t(static_cast<const float*>(logits), T, ld, plan, cs, dev_error,
                                dev, stream);
}

cudaError_t launch_combine(const float4* cs, const ShardPlan& plan, const void* logits,
                           pstat_dtype dt, int64_t T, int64_t V, int64_t ld,
                           const int64_t* labels, int64_t ignore_index, const float* target,
                           float* logprob, float* entropy, float* rowstats, int* dev_error,
                           cudaStream_t stream) {
    const int threads = kCombineWarps * 32;
    const unsigned grid = (unsigned)((T + kCombineWarps - 1) / kCombineWarps);
    if (dt == PSTAT_BF16)
        combine_kernel<uint16_t><<<grid, threads, 0, stream>>>(
            cs, plan, static_cast<const uint16_t*>(logits), T, V, ld, labels, ignore_index,
            target, logprob, entropy, rowstats, dev_error);
    else
        combine_kernel<float><<<grid, threads, 0, stream>>>(
            cs, plan, static_cast<const float*>(logits), T, V, ld, labels, ignore_index, target,
            logprob, entropy, rowstats, dev_error);
    return cudaGetLastError();
}

template <typename Ein, typename Eout>
static void launch_backward_t(const Ein* logits, int64_t T, int64_t V, int64_t ld,
                              const int64_t* labels, int64_t ignore_index, const float* weights,
                              const float* rowstats, Eout* out, int64_t ld_out, int* dev_error,
                              const DeviceInfo& dev, cudaStream_t stream, int64_t label_offset,
                              int64_t v_total) {
    // Segments per row: enough CTAs to fill the GPU many times over, each
    // streaming at least ~32K elements.
    int64_t segs = V / 32768;
    if (segs < 1) segs = 1;
    if (segs > 64) segs = 64;
    const int64_t grid = T * segs;
    backward_kernel<Ein, Eout><<<(unsigned)grid, kBwdThreads, 0, stream>>>(
        logits, V, ld, labels, ignore_index, weights, reinterpret_cast<const float2*>(rowstats),
        out, ld_out, (int)segs, label_offset, v_total, dev_error);
    (void)dev;
}

cudaError_t launch_backward(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                            int64_t ld, const int64_t* labels, int64_t ignore_index,
                            const float* weights, const float* rowstats, void* out,
                            pstat_dtype out_dt, int64_t ld_out, int* dev_error,
                            const DeviceInfo& dev, cudaStream_t stream, int64_t label_offset,
                            int64_t v_total) {
    if (v_total < 0) v_total = V;
    if (dt == PSTAT_BF16 && out_dt == PSTAT_BF16)
        launch_backward_t(static_cast<const uint16_t*>(logits), T, V, ld, labels, ignore_index,
                          weights, rowstats, static_cast<uint16_t*>(out), ld_out, dev_error, dev,
                          stream, label_offset, v_total);
    else if (dt == PSTAT_F32 && out_dt == PSTAT_BF16)
        launch_backward_t(static_cast<const float*>(logits), T, V, ld, labels, ignore_index,
                          weights, rowstats, static_cast<uint16_t*>(out), ld_out, dev_error, dev,
                          stream, label_offset, v_total);
    else
        launch_backward_t(static_cast<const float*>(logits), T, V, ld, labels, ignore_index,
                          weights, rowstats, static_cast<float*>(out), ld_out, dev_error, dev,
                          stream, label_offset, v_total);
    return cudaGetLastError();
}

}  // namespace pstat

namespace pstat {

template <typename Ein, typename Eout>
static void launch_logsoftmax_t(const Ein* logits, int64_t T, int64_t V, int64_t ld,
                                const float* rowstats, Eout* out, int64_t ld_out, int* dev_error,
                                cudaStream_t stream) {
    int64_t segs = V / 32768;
    if (segs < 1) segs = 1;
    if (segs > 64) segs = 64;
    logsoftmax_kernel<Ein, Eout><<<(unsigned)(T * segs), kBwdThreads, 0, stream>>>(
        logits, V, ld, reinterpret_cast<const float2*>(rowstats), out, ld_out, (int)segs, dev_error);
}

cudaError_t launch_logsoftmax(const void* logits, pstat_dtype dt, int64_t T, int64_t V, int64_t ld,
                              const float* rowstats, void* out, pstat_dtype out_dt, int64_t ld_out,
                              int* dev_error, cudaStream_t stream) {
    if (dt == PSTAT_BF16 && out_dt == PSTAT_BF16)
        launch_logsoftmax_t(static_cast<const uint16_t*>(logits), T, V, ld, rowstats,
                            static_cast<uint16_t*>(out), ld_out, dev_error, stream);
    else if (dt == PSTAT_BF16)
        launch_logsoftmax_t(static_cast<const uint16_t*>(logits), T, V, ld, rowstats,
                            static_cast<float*>(out), ld_out, dev_error, stream);
    else if (out_dt == PSTAT_BF16)
        launch_logsoftmax_t(static_cast<const float*>(logits), T, V, ld, rowstats,
                            static_cast<uint16_t*>(out), ld_out, dev_error, stream);
    else
        launch_logsoftmax_t(static_cast<const float*>(logits), T, V, ld, rowstats,
                            static_cast<float*>(out), ld_out, dev_error, stream);
    return cudaGetLastError();
}

}  // namespace pstat
