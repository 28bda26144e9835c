// chunk_math.cuh -- device arithmetic shared by the statistics kernels:
// the fixed chunk plan, the per-chunk reduction (bf16 and fp32), the
// fixed-order fold of chunk records into row statistics, and the element-wise
// gradient.  Every kernel that produces or consumes chunk statistics uses
// these same functions, so their results are bit-identical.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace pstat {

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
    static constexpr int kChunk = PSTAT_CHUNK_BF16;
    __device__ static uint16_t neg_inf() { return 0xFF80u; }
    __device__ static float to_float(uint16_t v) { return __uint_as_float((uint32_t)v << 16); }
    __device__ static uint4 neg_inf_vec() {
        return make_uint4(kBf16NegInf2, kBf16NegInf2, kBf16NegInf2, kBf16NegInf2);
    }
};
template <>
struct Elem<float> {
    static constexpr int kVec = 4;
    static constexpr int kChunk = PSTAT_CHUNK_F32;
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

// Maximum over the 32 lanes of a converged warp in one reduction (NaN inputs
// ignored, as fmaxf does; exact, so the order of the lanes does not matter).
__device__ __forceinline__ float warp_max(float m) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(m));
    return r;
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
//
// The exponent pass first runs without any clamp.  Only a -inf logit can make
// it produce NaN (e = 0 times a = -inf); then, and only then, the chunk is
// redone with every element raised to clamp_floor(m), below which e^(z - m)
// is 0 in fp32 anyway.  A chunk shorter than a full one, padded with -inf,
// takes the clamped pass directly.  Which pass a chunk takes depends only on
// its own values and length, so the result is still a fixed function of the
// chunk.
template <bool kClamp>
__device__ __forceinline__ void exp_sums_bf16(const uint4 (&q)[kVecPerLane], float m, float m2,
                                              float& s_out, float& u_out) {
    uint32_t fl2 = 0;
    if (kClamp) {
        const uint32_t f16 = bf16_round_down(clamp_floor(m));
        fl2 = f16 | (f16 << 16);
    }
    const uint64_t L2 = f2_pack(kLog2e, kLog2e);
    const uint64_t nm2 = f2_pack(-m2, -m2);
    uint64_t s0 = 0, s1 = 0, s2 = 0, s3 = 0, u0 = 0, u1 = 0, u2 = 0, u3 = 0;  // (+0, +0) pairs
    auto step = [&](uint32_t word, uint64_t& s, uint64_t& u) {
        const uint32_t w = kClamp ? bf2_max(word, fl2) : word;
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
    s_out = s;
    u_out = u;
}

// `len` is the chunk's length: load_chunk_regs pads a shorter chunk with -inf
// vectors, which would make the unclamped pass NaN, so such a chunk goes
// straight to the clamped one (the pass it would have ended in).  So does any
// chunk with `clamp_first`: without a -inf in the chunk the two passes give
// the same bits (every element the clamp raises has e = 0 either way), so the
// caller may choose by any rule.  *had_inf is set when a full chunk's
// unclamped pass came out NaN.
__device__ __forceinline__ float4 reduce_regs(const uint4 (&q)[kVecPerLane], uint16_t*,
                                              int len = PSTAT_CHUNK_BF16,
                                              bool clamp_first = false,
                                              bool* had_inf = nullptr) {
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
    float s = 0.f, u = NAN;
    const bool unclamped = len == PSTAT_CHUNK_BF16 && !clamp_first;
    if (unclamped) exp_sums_bf16<false>(q, m, m2, s, u);
    if (u != u) {  // warp-uniform: the butterfly agrees
        if (had_inf && unclamped) *had_inf = true;
        exp_sums_bf16<true>(q, m, m2, s, u);
    }
    return make_float4(m, s, u * kLn2, delta * kLn2);
}

// Same for fp32 chunks: 4-element vectors, two packed accumulators per lane.
__device__ __forceinline__ float4 reduce_regs(const uint4 (&q)[kVecPerLane], float*, int = 0,
                                              bool = true, bool* = nullptr) {
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


// Slot -> registers: lane L takes the 16-byte vectors L, L+32, ..., L+480 of
// the chunk; vectors past its end read as -inf.  A full chunk (the common
// case) needs no per-vector test.
template <typename E>
__device__ __forceinline__ void load_chunk_regs(const void* buf, int len, int lane,
                                                uint4 (&q)[kVecPerLane]) {
    const uint4* v = reinterpret_cast<const uint4*>(buf) + lane;
    constexpr int kVec = Elem<E>::kVec;
    const int nvec = (len + kVec - 1) / kVec;
    if (nvec == 32 * kVecPerLane) {
#pragma unroll
        for (int jj = 0; jj < kVecPerLane; ++jj) q[jj] = v[32 * jj];
    } else {
#pragma unroll
        for (int jj = 0; jj < kVecPerLane; ++jj)
            q[jj] = (lane + 32 * jj < nvec) ? v[32 * jj] : Elem<E>::neg_inf_vec();
    }
}

// ---------------------------------------------------------------------------
// Fixed-order fold of one row's chunk records, by one warp.
// A record (m, s, u, dr) holds its sums relative to the reference point
// m - dr.  Within a shard: M_s = max of its chunk maxima; each chunk moves to
// M_s with f = e^((m_c - M_s) - dr_c),
//     S_s = sum_c f s_c,   U_s = sum_c f (u_c + ((m_c - M_s) - dr_c) s_c),
// the sums taken as: lane L adds the shard's chunks L, L+32, ... (counted
// from the shard start) in ascending order, then the lanes are added by an
// xor butterfly.  Across shards, in ascending order, the same with the row
// maximum M.  Chunks or shards whose maximum is -inf (fully masked) are
// skipped.  The order depends only on the shard plan, and every lane ends
// with the same (M, S, U).
// ---------------------------------------------------------------------------
// Moves one shard's sums (ps, pu), relative to its maximum Ms, onto the row
// maximum M and adds them to the running row sums (S, U).  Shards are taken in
// ascending order; a shard whose maximum is -inf is skipped by the caller.
// This is the cross-shard step of fold_row_warp, which writes the same
// operations out in place (as a call there the compiler schedules the
// single-pass kernel's hot loop measurably worse); the two must stay
// identical, and the vocabulary-parallel tests compare their bits.
__device__ __forceinline__ void fold_shard(float Ms, float ps, float pu, float M, float& S,
                                           float& U) {
    const float dM = Ms - M;
    const float f = expf(dM);
    S = fmaf(ps, f, S);
    U = fmaf(f, fmaf(dM, ps, pu), U);
}

__device__ __forceinline__ float3 fold_row_warp(const float4* rec, const ShardPlan& plan,
                                                int lane) {
    // With one shard its maximum is the row maximum: no separate pass.
    float M = -INFINITY;
    if (plan.n_shards > 1) {
        for (int c = lane; c < plan.n_chunks; c += 32) M = fmaxf(M, rec[c].x);
        M = warp_max(M);
    }
    float S = 0.f, U = 0.f;
    if (plan.n_shards == 1 || M > -INFINITY) {
        for (int sh = 0; sh < plan.n_shards; ++sh) {
            const int c0 = plan.cum[sh], c1 = plan.cum[sh + 1];
            float Ms = -INFINITY;
            for (int c = c0 + lane; c < c1; c += 32) Ms = fmaxf(Ms, rec[c].x);
            Ms = warp_max(Ms);
            if (plan.n_shards == 1) M = Ms;
            if (Ms == -INFINITY) continue;
            float ps = 0.f, pu = 0.f;
            for (int c = c0 + lane; c < c1; c += 32) {
                const float4 r = rec[c];
                if (r.x == -INFINITY) continue;
                const float dm = (r.x - Ms) - r.w;
                const float f = expf(dm);
                ps = fmaf(r.y, f, ps);
                pu = fmaf(f, fmaf(dm, r.y, r.z), pu);
            }
#pragma unroll
            for (int off = 16; off; off >>= 1) {
                ps += __shfl_xor_sync(0xFFFFFFFFu, ps, off);
                pu += __shfl_xor_sync(0xFFFFFFFFu, pu, off);
            }
            const float dM = Ms - M;
            const float f = expf(dM);
            S = fmaf(ps, f, S);
            U = fmaf(f, fmaf(dM, ps, pu), U);
        }
    }
    return make_float3(M, S, U);
}

// ---------------------------------------------------------------------------
// Element-wise gradient helpers: 8 elements per 16-byte (bf16) or 32-byte
// (fp32) vector.
// ---------------------------------------------------------------------------
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

// Element-wise softmax for the gradient.  With m2 = RN(M log2e) and its exact
// residual delta = M log2e - m2 (one FMA),
//     e^(z - M - ln S) = 2^(RN(z log2e - m2)) * K,   K = 2^-(RN(ln S log2e + delta)),
// up to roundings, so an element costs one packed FMA and one exp2 -- the
// form of the chunk statistics -- and the row factor K (times -w) rides on
// the multiply the gradient needs anyway.  The row constants depend on
// (M, ln S, w) only, so every kernel that forms the gradient from the same
// row statistics produces the same bits.
struct GradRow {
    float m2;   // RN(M log2e)
    float K;    // 2^-(ln S log2e + delta)
    float nwK;  // -w K
    float w;
};
__device__ __forceinline__ GradRow grad_row(float M, float lnS, float w) {
    GradRow r;
    r.m2 = M * kLog2e;
    const float delta = fmaf(M, kLog2e, -r.m2);
    r.K = exp2f(-fmaf(lnS, kLog2e, delta));
    r.nwK = -w * r.K;
    r.w = w;
    return r;
}

// e_i = 2^(RN(x_i log2e - m2)) for 8 elements.
__device__ __forceinline__ void exp8(const float (&x)[8], float m2, float (&e)[8]) {
    const uint64_t l2e = f2_pack(kLog2e, kLog2e);
    const uint64_t nm2 = f2_pack(-m2, -m2);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float a0, a1;
        f2_unpack(f2_fma(f2_pack(x[2 * i], x[2 * i + 1]), l2e, nm2), a0, a1);
        e[2 * i] = ex2_approx(a0);
        e[2 * i + 1] = ex2_approx(a1);
    }
}

// g_i = -w p_i = e_i (-w K) for 8 elements (the label column is fixed by the caller).
__device__ __forceinline__ void grad8(const float (&e)[8], const GradRow& r, float (&g)[8]) {
    const uint64_t k = f2_pack(r.nwK, r.nwK);
#pragma unroll
    for (int i = 0; i < 4; ++i) f2_unpack(f2_mul(f2_pack(e[2 * i], e[2 * i + 1]), k), g[2 * i], g[2 * i + 1]);
}

// The label column: w (1 - p_y) with p_y = e_y K.
__device__ __forceinline__ float grad_label(float e_y, const GradRow& r) {
    return fmaf(-r.w, e_y * r.K, r.w);
}

}  // namespace pstat
