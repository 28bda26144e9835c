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
// Per chunk (m = chunk maximum, L = log2(e) rounded to fp32):
//   m2 = RN(m L), delta = m L - m2 (exact, by one FMA),
//   a_i = RN(z_i L - m2)      one packed FMA per pair of elements,
//   e_i = 2^a_i               (MUFU ex2),
//   s = sum e_i,  u = ln2 * sum e_i a_i.
// Since a_i = (z_i - m) L + delta up to its own rounding, s and u are the sum
// of exponentials and the entropy-weighted sum relative to the reference
// point r = m - delta ln2 (in natural units).  The record is
// (m, s, u, delta ln2); the combine moves it to any common maximum M with
// the factor e^((m - M) - delta ln2).  This costs one FMA per element where
// the direct form z - m, then times log2(e), costs two.
// ---------------------------------------------------------------------------
constexpr int kWarps = 12;
constexpr int kStages = 2;
constexpr int kSlotBytes = 8192;
constexpr int kVecPerLane = kSlotBytes / 16 / 32;  // 16
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any legal copy
constexpr float kLn2 = 0.6931471805599453f;

static_assert(PSTAT_CHUNK_BF16 * 2 == kSlotBytes, "bf16 chunk must fill one slot");
static_assert(PSTAT_CHUNK_F32 * 4 == kSlotBytes, "fp32 chunk must fill one slot");

constexpr size_t chunk_stats_smem_bytes() {
    return (size_t)kWarps * kStages * kSlotBytes + (size_t)kWarps * kStages * sizeof(uint64_t);
}

template <typename E>
struct Elem;
template <>
struct Elem<uint16_t> {  // bf16 bit patterns
    static constexpr int kVec = 8;  // elements per 16-byte vector
    __device__ static uint16_t neg_inf() { return 0xFF80u; }
    __device__ static float to_float(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }
    __device__ static uint4 neg_inf_vec() {
        return make_uint4(kBf16NegInf2, kBf16NegInf2, kBf16NegInf2, kBf16NegInf2);
    }
};
template <>
struct Elem<float> {
    static constexpr int kVec = 4;
    __device__ static float neg_inf() { return -INFINITY; }
    __device__ static float to_float(float v) { return v; }
    __device__ static uint4 neg_inf_vec() {
        const uint32_t n = 0xFF800000u;
        return make_uint4(n, n, n, n);
    }
};

// Column span [start, start + len) of chunk g of every row.
__device__ __forceinline__ void chunk_span(const ShardPlan& p, int g, int64_t& start, int& len) {
    int s = 0;
    while (p.cum[s + 1] <= g) ++s;
    start = p.bounds[s] + (int64_t)(g - p.cum[s]) * p.chunk;
    const int64_t end = min(start + (int64_t)p.chunk, p.bounds[s + 1]);
    len = (int)(end - start);
}

// Largest bf16 value <= x (x finite): truncating the float rounds toward
// zero, so negative values with dropped bits step one ulp further down.
__device__ __forceinline__ uint32_t bf16_round_down(float x) {
    const uint32_t b = __float_as_uint(x);
    uint32_t h = b >> 16;
    if ((b & 0x80000000u) && (b & 0xFFFFu)) h += 1;
    return h;
}

// Lower clamp for the exponential pass.  Every element below it has
// e^(z-m) == 0 in fp32 anyway; clamping keeps the exponent finite so that
// -inf logits add exactly 0 to u instead of 0 * (-inf) = NaN.
__device__ __forceinline__ float clamp_floor(float m) {
    return m - fmaxf(1024.f, fabsf(m) * 0.0625f);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ float warp_max(float m) {
#pragma unroll
    for (int off = 16; off; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    return m;
}

__device__ __forceinline__ float hsum2(uint64_t p) {
    float lo, hi;
    f2_unpack(p, lo, hi);
    return lo + hi;
}

// Statistics of one chunk held in registers (bf16).  Lane-local sums run over
// the lane's vectors in ascending order with one packed accumulator per
// 32-bit word; the four are added in a fixed tree, then lanes by an xor
// butterfly (which leaves the same bits in every lane).
__device__ __forceinline__ float4 reduce_regs(const uint4 (&q)[kVecPerLane], uint16_t*) {
    uint32_t a0 = q[0].x, a1 = q[0].y, a2 = q[0].z, a3 = q[0].w;
#pragma unroll
    for (int j = 1; j < kVecPerLane; ++j) {
        a0 = bf2_max(a0, q[j].x);
        a1 = bf2_max(a1, q[j].y);
        a2 = bf2_max(a2, q[j].z);
        a3 = bf2_max(a3, q[j].w);
    }
    const uint32_t a = bf2_max(bf2_max(a0, a1), bf2_max(a2, a3));
    const float m = warp_max(fmaxf(bf2_lo(a), bf2_hi(a)));
    if (m == -INFINITY) return make_float4(m, 0.f, 0.f, 0.f);  // fully masked chunk
    const float m2 = m * kLog2e;
    const float delta = fmaf(m, kLog2e, -m2);
    const uint32_t f16 = bf16_round_down(clamp_floor(m));
    const uint32_t fl2 = f16 | (f16 << 16);
    const uint64_t L2 = f2_pack(kLog2e, kLog2e);
    const uint64_t nm2 = f2_pack(-m2, -m2);
    uint64_t s0 = 0, s1 = 0, s2 = 0, s3 = 0, u0 = 0, u1 = 0, u2 = 0, u3 = 0;  // (+0, +0) pairs
    auto step = [&](uint32_t word, uint64_t& s, uint64_t& u) {
        const uint32_t w = bf2_max(word, fl2);
        const uint64_t a = f2_fma(f2_pack(bf2_lo(w), bf2_hi(w)), L2, nm2);
        float a0_, a1_;
        f2_unpack(a, a0_, a1_);
        const uint64_t e = f2_pack(ex2_approx(a0_), ex2_approx(a1_));
        s = f2_add(s, e);
        u = f2_fma(e, a, u);
    };
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
        step(q[j].x, s0, u0);
        step(q[j].y, s1, u1);
        step(q[j].z, s2, u2);
        step(q[j].w, s3, u3);
    }
    float s = (hsum2(s0) + hsum2(s1)) + (hsum2(s2) + hsum2(s3));
    float u = (hsum2(u0) + hsum2(u1)) + (hsum2(u2) + hsum2(u3));
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
        u += __shfl_xor_sync(0xFFFFFFFFu, u, off);
    }
    return make_float4(m, s, u * kLn2, delta * kLn2);
}

// Same for fp32 chunks: 4-element vectors, two packed accumulators per lane.
__device__ __forceinline__ float4 reduce_regs(const uint4 (&q)[kVecPerLane], float*) {
    float a0 = -INFINITY, a1 = -INFINITY;
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
        a0 = max3(a0, __uint_as_float(q[j].x), __uint_as_float(q[j].y));
        a1 = max3(a1, __uint_as_float(q[j].z), __uint_as_float(q[j].w));
    }
    const float m = warp_max(fmaxf(a0, a1));
    if (m == -INFINITY) return make_float4(m, 0.f, 0.f, 0.f);
    const float m2 = m * kLog2e;
    const float delta = fmaf(m, kLog2e, -m2);
    const float fl = clamp_floor(m);
    const uint64_t L2 = f2_pack(kLog2e, kLog2e);
    const uint64_t nm2 = f2_pack(-m2, -m2);
    uint64_t s0 = 0, s1 = 0, u0 = 0, u1 = 0;
    auto step = [&](uint32_t x, uint32_t y, uint64_t& s, uint64_t& u) {
        const uint64_t a = f2_fma(f2_pack(fmaxf(__uint_as_float(x), fl), fmaxf(__uint_as_float(y), fl)),
                                  L2, nm2);
        float a0_, a1_;
        f2_unpack(a, a0_, a1_);
        const uint64_t e = f2_pack(ex2_approx(a0_), ex2_approx(a1_));
        s = f2_add(s, e);
        u = f2_fma(e, a, u);
    };
#pragma unroll
    for (int j = 0; j < kVecPerLane; ++j) {
        step(q[j].x, q[j].y, s0, u0);
        step(q[j].z, q[j].w, s1, u1);
    }
    float s = hsum2(s0) + hsum2(s1);
    float u = hsum2(u0) + hsum2(u1);
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
        u += __shfl_xor_sync(0xFFFFFFFFu, u, off);
    }
    return make_float4(m, s, u * kLn2, delta * kLn2);
}

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

    auto locate = [&](int64_t i, const E*& src, int& len) -> bool {
        const int64_t t = i / plan.n_chunks;
        const int g = (int)(i - t * plan.n_chunks);
        int64_t start;
        chunk_span(plan, g, start, len);
        src = logits + t * ld + start;
        return ((reinterpret_cast<uintptr_t>(src) & 15u) == 0) &&
               ((((size_t)len * sizeof(E)) & 15u) == 0);
    };
    auto issue = [&](int64_t i, int slot) {
        const E* src;
        int len;
        if (locate(i, src, len) && lane == 0) {
            const uint32_t bytes = (uint32_t)len * (uint32_t)sizeof(E);
            mbar_arrive_expect_tx(&bars[slot], bytes);
            bulk_g2s_evict_first(slots + (size_t)slot * kSlotBytes, src, bytes, &bars[slot],
                                 policy);
        }
    };

    const int64_t prologue = n < kStages ? n : kStages;
    for (int64_t j = 0; j < prologue; ++j) issue(i0 + j, (int)j);

    uint32_t phase = 0;  // parity bit per slot, flipped after each bulk completion
    int64_t j = 0;
    bool timed_out = false;
    for (; j < n; ++j) {
        const int slot = (int)(j % kStages);
        E* buf = reinterpret_cast<E*>(slots + (size_t)slot * kSlotBytes);
        const E* src;
        int len;
        if (locate(i0 + j, src, len)) {
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
        // Slot -> registers; vectors past the chunk end read as -inf.
        constexpr int kVec = Elem<E>::kVec;
        const int nvec = (len + kVec - 1) / kVec;
        const uint4* v = reinterpret_cast<const uint4*>(buf);
        uint4 q[kVecPerLane];
#pragma unroll
        for (int jj = 0; jj < kVecPerLane; ++jj) {
            const int k = lane + 32 * jj;
            q[jj] = (k < nvec) ? v[k] : Elem<E>::neg_inf_vec();
        }
        __syncwarp();
        fence_proxy_async_smem();  // our reads of the slot precede the next bulk write into it
        if (j + kStages < n) issue(i0 + j + kStages, slot);
        const float4 r = reduce_regs(q, (E*)nullptr);
        if (lane == 0) out[i0 + j] = r;
    }
    if (timed_out) {
        if (lane == 0 && dev_error) atomicOr(dev_error, PSTAT_DEV_TIMEOUT);
        // Drain copies still in flight into this CTA's shared memory before leaving.
        const int64_t last = (j + kStages < n) ? j + kStages : n;
        for (int64_t k = j; k < last; ++k) {
            const int slot = (int)(k % kStages);
            const E* src;
            int len;
            if (locate(i0 + k, src, len)) {
                mbar_wait_bounded(&bars[slot], (phase >> slot) & 1u, kWaitLimitNs);
                phase ^= 1u << slot;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// K-B: fixed-order combine, one thread per row.
// A chunk record (m, s, u, dr) holds its sums relative to the reference point
// m - dr (dr = 0 when the producer shifted by m itself).  Within a shard:
// M_s = max of its chunk maxima, then its chunks in ascending order are moved
// to M_s and summed, with f = e^((m_c - M_s) - dr_c):
//     S_s = sum_c f s_c,   U_s = sum_c f (u_c + ((m_c - M_s) - dr_c) s_c).
// Across shards: the same with the row maximum M, shards in ascending order.
// Chunks or shards whose maximum is -inf (fully masked) are skipped.
// The CTA first copies its rows' records into shared memory with coalesced
// loads (when they fit), so each thread's sequential fold reads on-chip data.
// ---------------------------------------------------------------------------
constexpr int kCombineRows = 32;     // rows per CTA
constexpr int kCombineThreads = 128;
constexpr int kCombineSmemRecords = 3072;  // 48 KB of float4

__device__ __forceinline__ float4 fold_row(const float4* c, const ShardPlan& plan) {
    float M = -INFINITY;
    for (int g = 0; g < plan.n_chunks; ++g) M = fmaxf(M, c[g].x);
    float S = 0.f, U = 0.f;
    if (M > -INFINITY) {
        for (int sh = 0; sh < plan.n_shards; ++sh) {
            float Ms = -INFINITY;
            for (int g = plan.cum[sh]; g < plan.cum[sh + 1]; ++g) Ms = fmaxf(Ms, c[g].x);
            if (Ms == -INFINITY) continue;
            float Ss = 0.f, Us = 0.f;
            for (int g = plan.cum[sh]; g < plan.cum[sh + 1]; ++g) {
                const float4 r = c[g];
                if (r.x == -INFINITY) continue;
                const float dm = (r.x - Ms) - r.w;
                const float f = expf(dm);
                Ss = fmaf(r.y, f, Ss);
                Us = fmaf(f, fmaf(dm, r.y, r.z), Us);
            }
            const float dM = Ms - M;
            const float f = expf(dM);
            S = fmaf(Ss, f, S);
            U = fmaf(f, fmaf(dM, Ss, Us), U);
        }
    }
    return make_float4(M, S, U, 0.f);
}

template <typename E>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float4* __restrict__ cs, const __grid_constant__ ShardPlan plan,
                   const E* __restrict__ logits, int64_t T, int64_t V, int64_t ld,
                   const int64_t* __restrict__ labels, int64_t ignore_index,
                   const float* __restrict__ target, float* __restrict__ logprob,
                   float* __restrict__ entropy, float* __restrict__ rowstats,
                   int* __restrict__ dev_error) {
    __shared__ float4 stage[kCombineSmemRecords];
    const int64_t t0 = (int64_t)blockIdx.x * kCombineRows;
    const int64_t rows = min((int64_t)kCombineRows, T - t0);
    const int nc = plan.n_chunks;
    const bool staged = (int64_t)kCombineRows * nc <= kCombineSmemRecords;
    if (staged) {
        const int64_t n = rows * nc;
        const float4* src = cs + t0 * nc;
        for (int64_t i = threadIdx.x; i < n; i += kCombineThreads) stage[i] = src[i];
        __syncthreads();
    }
    if (threadIdx.x >= rows) return;
    const int64_t t = t0 + threadIdx.x;
    const float4 st = fold_row(staged ? stage + (int64_t)threadIdx.x * nc : cs + t * nc, plan);
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
constexpr int kBwdThreads = 256;
constexpr int kBwdUnroll = 4;

template <typename E>
struct Load8;
template <>
struct Load8<uint16_t> {
    __device__ static void run(const uint16_t* p, float (&x)[8]) {
        const uint4 q = __ldcs(reinterpret_cast<const uint4*>(p));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = bf2_lo(w[i]);
            x[2 * i + 1] = bf2_hi(w[i]);
        }
    }
};
template <>
struct Load8<float> {
    __device__ static void run(const float* p, float (&x)[8]) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
        const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
};
template <typename E>
struct Store8;
template <>
struct Store8<uint16_t> {
    __device__ static void run(uint16_t* p, const float (&g)[8]) {
        uint4 q;
        q.x = bf2_pack_rn(g[0], g[1]);
        q.y = bf2_pack_rn(g[2], g[3]);
        q.z = bf2_pack_rn(g[4], g[5]);
        q.w = bf2_pack_rn(g[6], g[7]);
        __stcs(reinterpret_cast<uint4*>(p), q);
    }
};
template <>
struct Store8<float> {
    __device__ static void run(float* p, const float (&g)[8]) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(g[0], g[1], g[2], g[3]));
        __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(g[4], g[5], g[6], g[7]));
    }
};
__device__ __forceinline__ uint16_t out_cast(float g, uint16_t*) {
    return (uint16_t)(bf2_pack_rn(g, 0.f) & 0xFFFFu);
}
__device__ __forceinline__ float out_cast(float g, float*) { return g; }

// p = e^(z - M - ln S) for 8 elements.
__device__ __forceinline__ void prob8(const float (&x)[8], float M, float log2S, float (&p)[8]) {
    const uint64_t negM = f2_pack(-M, -M);
    const uint64_t l2e = f2_pack(kLog2e, kLog2e);
    const uint64_t nl2s = f2_pack(-log2S, -log2S);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint64_t d = f2_add(f2_pack(x[2 * i], x[2 * i + 1]), negM);
        float a0, a1;
        f2_unpack(f2_fma(d, l2e, nl2s), a0, a1);
        p[2 * i] = ex2_approx(a0);
        p[2 * i + 1] = ex2_approx(a1);
    }
}

template <typename Ein, typename Eout>
__global__ void __launch_bounds__(kBwdThreads)
    backward_kernel(const Ein* __restrict__ logits, int64_t V, int64_t ld,
                    const int64_t* __restrict__ labels, int64_t ignore_index,
                    const float* __restrict__ weights, const float2* __restrict__ rowstats,
                    Eout* __restrict__ out, int64_t ld_out, int segs, int* __restrict__ dev_error) {
    const int64_t t = blockIdx.x / segs;
    const int seg = (int)(blockIdx.x - t * segs);
    const int64_t nv_row = V >> 3;  // whole 8-element groups in the row
    const int64_t c0 = (nv_row * seg / segs) << 3;
    const int64_t c1 = (seg == segs - 1) ? V : ((nv_row * (seg + 1) / segs) << 3);
    const Ein* zin = logits + t * ld;
    Eout* zout = out + t * ld_out;

    const int64_t y = labels ? labels[t] : ignore_index;
    const float w = weights ? weights[t] : 1.f;
    int mode;  // 0: zero row, 1: NaN row, 2: compute
    float M = 0.f, log2S = 0.f;
    if (y == ignore_index || w == 0.f) {
        mode = 0;
    } else {
        const float2 rs = rowstats[t];
        if (y < 0 || y >= V || !(rs.x > -INFINITY) || !(rs.y == rs.y)) {
            mode = 1;
            if (seg == 0 && threadIdx.x == 0 && dev_error)
                atomicOr(dev_error, (y < 0 || y >= V) ? PSTAT_DEV_BAD_LABEL : PSTAT_DEV_EMPTY_ROW);
        } else {
            mode = 2;
            M = rs.x;
            log2S = rs.y * kLog2e;
        }
    }
    const float fill = (mode == 0) ? 0.f : NAN;
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(zin + c0) & 15u) == 0) &&
                        ((reinterpret_cast<uintptr_t>(zout + c0) & 15u) == 0);
    const int64_t nv = vec_ok ? (c1 - c0) >> 3 : 0;
    const float negw = -w;

    for (int64_t base = 0; base < nv; base += (int64_t)kBwdThreads * kBwdUnroll) {
        float x[kBwdUnroll][8];
        int64_t col[kBwdUnroll];
#pragma unroll
        for (int k = 0; k < kBwdUnroll; ++k) {
            const int64_t i = base + (int64_t)k * kBwdThreads + threadIdx.x;
            col[k] = (i < nv) ? c0 + (i << 3) : -1;
            if (mode == 2 && col[k] >= 0) Load8<Ein>::run(zin + col[k], x[k]);
        }
#pragma unroll
        for (int k = 0; k < kBwdUnroll; ++k) {
            if (col[k] < 0) continue;
            float g[8];
            if (mode == 2) {
                float p[8];
                prob8(x[k], M, log2S, p);
                const uint64_t nw = f2_pack(negw, negw);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    f2_unpack(f2_mul(f2_pack(p[2 * i], p[2 * i + 1]), nw), g[2 * i], g[2 * i + 1]);
                const int64_t r = y - col[k];
                if (r >= 0 && r < 8) {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (e == r) g[e] = fmaf(negw, p[e], w);  // w (1 - p_y)
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
            const float a = fmaf(x - M, kLog2e, -log2S);
            const float p = ex2_approx(a);
            g = (c == y) ? fmaf(negw, p, w) : negw * p;
        } else {
            g = fill;
        }
        zout[c] = out_cast(g, zout);
    }
}

// ---------------------------------------------------------------------------
// Launchers.
// ---------------------------------------------------------------------------
template <typename E>
static cudaError_t launch_chunk_stats_t(const E* logits, int64_t T, int64_t ld,
                                        const ShardPlan& plan, float4* cs, int* dev_error,
                                        const DeviceInfo& dev, cudaStream_t stream) {
    static std::atomic<bool> configured[64];
    int d = 0;
    cudaGetDevice(&d);
    const size_t smem = chunk_stats_smem_bytes();
    if (d >= 64 || !configured[d].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(chunk_stats_kernel<E>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (d < 64) configured[d].store(true, std::memory_order_release);
    }
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
    const int threads = kCombineThreads;
    const unsigned grid = (unsigned)((T + kCombineRows - 1) / kCombineRows);
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
                              const DeviceInfo& dev, cudaStream_t stream) {
    // Segments per row: enough CTAs to fill the GPU many times over, each
    // streaming at least ~32K elements.
    int64_t segs = V / 32768;
    if (segs < 1) segs = 1;
    if (segs > 64) segs = 64;
    const int64_t grid = T * segs;
    backward_kernel<Ein, Eout><<<(unsigned)grid, kBwdThreads, 0, stream>>>(
        logits, V, ld, labels, ignore_index, weights, reinterpret_cast<const float2*>(rowstats),
        out, ld_out, (int)segs, dev_error);
    (void)dev;
}

cudaError_t launch_backward(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                            int64_t ld, const int64_t* labels, int64_t ignore_index,
                            const float* weights, const float* rowstats, void* out,
                            pstat_dtype out_dt, int64_t ld_out, int* dev_error,
                            const DeviceInfo& dev, cudaStream_t stream) {
    if (dt == PSTAT_BF16 && out_dt == PSTAT_BF16)
        launch_backward_t(static_cast<const uint16_t*>(logits), T, V, ld, labels, ignore_index,
                          weights, rowstats, static_cast<uint16_t*>(out), ld_out, dev_error, dev,
                          stream);
    else if (dt == PSTAT_F32 && out_dt == PSTAT_BF16)
        launch_backward_t(static_cast<const float*>(logits), T, V, ld, labels, ignore_index,
                          weights, rowstats, static_cast<uint16_t*>(out), ld_out, dev_error, dev,
                          stream);
    else
        launch_backward_t(static_cast<const float*>(logits), T, V, ld, labels, ignore_index,
                          weights, rowstats, static_cast<float*>(out), ld_out, dev_error, dev,
                          stream);
    return cudaGetLastError();
}

}  // namespace pstat
