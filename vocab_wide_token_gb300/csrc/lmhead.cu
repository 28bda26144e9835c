// lmhead.cu -- fused lm_head on the 5th-generation tensor cores.
//
// Forward: logits z = hidden W^T are produced tile by tile (128 tokens x 256
// vocabulary rows, K = d in steps of 64) by tcgen05.mma into tensor memory
// and folded straight into the per-(token, 4096-column chunk) statistics
// (m, s, u) that the unfused path also produces; the logits never reach
// global memory.  The fixed-order combine kernel then gives logprob, entropy
// and (M, ln S).
//
// Backward, per 8192-column vocabulary chunk c (the chunked lm_head of TRL PR
// #6949 "ZeroSyncGRPOTrainer": GEMMs in a 16-bit dtype, accumulation in fp32
// buffers):
//   1. recompute the chunk's logits tile by tile and turn them on chip into
//      g = w (onehot(y) - e^(z - M - ln S)), stored as fp16 twice: G [T, Vc]
//      and its transpose Gt [Vc, T];
//   2. dhidden += G W_c        (A = G, B = W_c^T, both K-major fp16);
//   3. dW[c]   += Gt hidden    (A = Gt, B = hidden^T, both K-major fp16).
// fp16 (11-bit significand) keeps the gradient operand within ~3e-4 relative
// where bf16 would give ~2e-3; hidden and W convert to fp16 exactly while
// 2^-14 <= |x| <= 65504 (values above flag PSTAT_DEV_RANGE).
//
// One warp-specialised persistent GEMM kernel serves every step (192
// threads, one CTA per SM):
//   warp 0     TMA producer: 2-D tiled loads of A (128 x 64) and B (256 x 64)
//              k-blocks into a 4-stage shared-memory ring (128-byte swizzle)
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators)
//              and issues tcgen05.mma (M=128, N=256, K=16) from one thread
//   warps 2-5  epilogue: one thread per output row reads its accumulator row
//              from TMEM (tcgen05.ld.32x32b) and hands it to the epilogue
//              policy (statistics, gradient tile, or fp32 accumulation)
// Work is split into units of consecutive N tiles that one CTA processes in
// order (8 tiles = one 2048-column statistics chunk in the forward, 1
// elsewhere); units are ordered in groups of M tiles (32; 16 in the
// accumulation GEMMs) so the A slice they share stays in L2.
// There is no split-K: each output element is a fixed-order K reduction.
// All waits are bounded; a timeout sets PSTAT_DEV_TIMEOUT and the CTA winds
// down, draining its copies and MMAs before freeing tensor memory.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pstat {
namespace lm {

constexpr int BM = 128;            // output rows per tile (MMA M, TMEM lanes)
constexpr int BN = 256;            // output columns per tile (MMA N)
constexpr int BK = 64;             // K per stage: 64 x 16-bit = one 128-byte swizzle row
constexpr int UK = 16;             // K per tcgen05.mma of kind::f16
constexpr int STAGES = 4;
// Statistics chunk of the fused forward: 2048 vocabulary columns (8 tiles),
// folded in ascending tile order by one CTA.  Half the 4096 of the logits
// path: at V = 151,936 a 16-tile unit leaves some SMs 32 units (512 tiles)
// against an average of 500; 8-tile units cap that at 504.
constexpr int LM_CHUNK = 2048;
constexpr int STATS_TILES = LM_CHUNK / BN;
constexpr int VC = 8192;           // backward vocabulary chunk (columns staged as G / Gt)
constexpr int M_GROUP = 32;        // M tiles sharing the L2-resident slice of A
// The accumulation GEMMs (K = 8192 or T) stream a longer A slice per tile;
// 16-tile groups measured about 1% faster there than 32 (8 and 64: slower).
constexpr int ACC_M_GROUP = 16;
constexpr int THREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;   // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;      // double-buffered accumulator
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr int QD = 4;  // depth of the claimed-unit queue (dynamic scheduling)

struct Smem {
    // Offsets inside the 1024-byte aligned dynamic shared memory block.
    static constexpr uint32_t a = 0;
    static constexpr uint32_t b = a + STAGES * A_BYTES;
    static constexpr uint32_t bars = b + STAGES * B_BYTES;
    // full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, uq_full[QD], uq_empty[QD]
    static constexpr uint32_t n_bars = 2 * STAGES + 4 + 1 + 2 * QD;
    static constexpr uint32_t tmem_slot = bars + n_bars * 8;
    static constexpr uint32_t uq = tmem_slot + 16;  // int[QD]: claimed unit ids
    static constexpr uint32_t total = uq + QD * 4;
};
constexpr size_t SMEM_BYTES = Smem::total + 1024;  // + alignment slack

struct GemmGeo {
    int m_tiles, n_tiles, k_blocks;
    int tiles_per_unit;   // consecutive N tiles one CTA processes in order
    int units_per_m;      // ceil(n_tiles / tiles_per_unit)
    int64_t n_units;      // m_tiles * units_per_m
    int b_row0;           // first B row (tensor-map coordinate) of N tile 0
    int m_group;          // M tiles per group: units run M-fastest within a group
};

__host__ __device__ inline void unit_coords(const GemmGeo& g, int64_t u, int& m, int& un) {
    const int64_t per_group = (int64_t)g.m_group * g.units_per_m;
    const int grp = (int)(u / per_group);
    const int64_t rem = u - (int64_t)grp * per_group;
    int mg = g.m_tiles - grp * g.m_group;
    if (mg > g.m_group) mg = g.m_group;
    un = (int)(rem / mg);
    m = grp * g.m_group + (int)(rem % mg);
}

__device__ __forceinline__ int unit_tiles(const GemmGeo& g, int un) {
    const int nt = g.n_tiles - un * g.tiles_per_unit;
    return nt < g.tiles_per_unit ? nt : g.tiles_per_unit;
}

// One launch runs up to two GEMMs with the same epilogue type: units
// [0, n0) belong to problem 0, [n0, total) to problem 1.  With a claim counter
// (zeroed before the launch), CTAs take units in index order with atomicAdd,
// so a CTA that finishes early takes more; without one, unit u goes to CTA
// u mod gridDim.x.  Either way each tile has exactly one CTA computing it over
// K in a fixed order, so the results do not depend on the schedule.
template <class Epi>
struct Problem {
    CUtensorMap a, b;
    GemmGeo g;
    Epi epi;
};
template <class Epi>
struct Problems {
    Problem<Epi> p[2];
    int64_t n0, total;
    int* counter;  // device int, or nullptr for the static schedule
};

// Instruction descriptor for fp16 operands (A and B both f16, D fp32).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ---------------------------------------------------------------------------
// Epilogue policies.  Each has a per-thread State and three hooks called by
// the epilogue warps: unit_begin, tile (the accumulator of one tile is ready
// in tensor memory at `taddr`, lane = this thread's output row) and
// unit_end.
// ---------------------------------------------------------------------------

// Forward statistics: folds each 256-column tile into running (m, s, u) for
// its 4096-column chunk and records the target logit.
struct StatsEpi {
    int64_t T, V;
    int n_chunks;
    const int64_t* labels;
    int64_t ignore_index;
    float4* chunk_stats;
    float* target;

    struct State {
        int64_t t, y;
        bool valid;
        float mc, sc, uc;
    };

    __device__ void unit_begin(State& st, int m, int /*un*/, int row) const {
        st.t = (int64_t)m * BM + row;
        st.valid = st.t < T;
        st.y = (st.valid && labels) ? labels[st.t] : ignore_index;
        st.mc = -INFINITY;
        st.sc = 0.f;
        st.uc = 0.f;
    }

    // Folds tile statistics (mj, sj, uj) into the running chunk statistics.
    __device__ static void fold(State& st, float mj, float sj, float uj) {
        if (st.mc == -INFINITY) {
            st.mc = mj;
            st.sc = sj;
            st.uc = uj;
            return;
        }
        if (mj > st.mc) {
            const float dm = st.mc - mj;
            const float r = expf(dm);
            st.uc = r * fmaf(dm, st.sc, st.uc) + uj;
            st.sc = fmaf(r, st.sc, sj);
            st.mc = mj;
        } else {
            const float dm = mj - st.mc;
            const float r = expf(dm);
            st.sc = fmaf(r, sj, st.sc);
            st.uc = fmaf(r, fmaf(dm, sj, uj), st.uc);
        }
    }

    __device__ void tile(State& st, uint32_t taddr, int /*m*/, int n, int /*row*/) const {
        const int64_t col0 = (int64_t)n * BN;
        const int64_t left = V - col0;
        const int ncols = left < BN ? (int)left : BN;
        // pass 1: row maximum over the tile
        float mx = -INFINITY;
        for (int p = 0; p < BN / 32; ++p) {
            if (p * 32 >= ncols) break;
            float v[32];
            tmem_ld32(taddr + p * 32, v);
            tmem_ld_wait();
            if (p * 32 + 32 <= ncols) {
#pragma unroll
                for (int i = 0; i < 32; ++i) mx = fmaxf(mx, v[i]);
            } else {
                for (int i = 0; i < 32; ++i)
                    if (p * 32 + i < ncols) mx = fmaxf(mx, v[i]);
            }
        }
        // pass 2: sum e^(z - mx) and sum e^(z - mx)(z - mx), pairs in f32x2
        const uint64_t negm = f2_pack(-mx, -mx);
        const uint64_t l2e = f2_pack(kLog2e, kLog2e);
        uint64_t s2 = 0, u2 = 0;
        const int64_t yl = st.y - col0;
        for (int p = 0; p < BN / 32; ++p) {
            if (p * 32 >= ncols) break;
            float v[32];
            tmem_ld32(taddr + p * 32, v);
            tmem_ld_wait();
            if (st.valid && yl >= p * 32 && yl < p * 32 + 32 && yl < ncols) {
                float zy = 0.f;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (yl == p * 32 + i) zy = v[i];
                target[st.t] = zy;
            }
            if (p * 32 + 32 > ncols) {  // columns past V: e^(-1024) == 0 exactly
                for (int i = 0; i < 32; ++i)
                    if (p * 32 + i >= ncols) v[i] = mx - 1024.f;
            }
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
                const uint64_t dd = f2_add(f2_pack(v[i], v[i + 1]), negm);
                float a0, a1;
                f2_unpack(f2_mul(dd, l2e), a0, a1);
                const uint64_t e = f2_pack(ex2_approx(a0), ex2_approx(a1));
                s2 = f2_add(s2, e);
                u2 = f2_fma(e, dd, u2);
            }
        }
        float sa, sb, ua, ub;
        f2_unpack(s2, sa, sb);
        f2_unpack(u2, ua, ub);
        fold(st, mx, sa + sb, ua + ub);
    }

    __device__ void unit_end(State& st, int /*m*/, int un, int /*row*/) const {
        if (st.valid) chunk_stats[st.t * n_chunks + un] = make_float4(st.mc, st.sc, st.uc, 0.f);
    }
};

// Backward step 1: the recomputed logits tile becomes the gradient tile
// g = w (onehot(y) - e^(z - M - ln S)), written as fp16 to G [rows, ldg]
// (row-major) and Gt [cols, ldgt] (its transpose).  Rows past T, columns
// past V, ignored rows and zero-weight rows are written as +0.
struct GradEpi {
    int64_t T, V;
    int64_t c0;            // first vocabulary column of this chunk
    const int64_t* labels;
    int64_t ignore_index;
    const float* weights;
    const float2* rowstats;
    __half* G;
    int64_t ldg;
    __half* Gt;
    int64_t ldgt;
    int* dev_error;

    struct State {
        int64_t t, y;
        bool live;
        float M, log2S, w;
    };

    __device__ void unit_begin(State& st, int m, int /*un*/, int row) const {
        st.t = (int64_t)m * BM + row;
        st.live = false;
        st.y = ignore_index;
        st.M = 0.f;
        st.log2S = 0.f;
        st.w = 0.f;
        if (st.t < T) {
            st.y = labels ? labels[st.t] : ignore_index;
            st.w = weights ? weights[st.t] : 1.f;
            if (st.y != ignore_index && st.w != 0.f) {
                const float2 rs = rowstats[st.t];
                st.M = rs.x;
                st.log2S = rs.y * kLog2e;
                st.live = true;
                if (st.y < 0 || st.y >= V || !(rs.x > -INFINITY) || !(rs.y == rs.y)) {
                    st.live = false;  // undefined row: flagged, written as zeros
                    if (dev_error && c0 == 0)
                        atomicOr(dev_error, (st.y < 0 || st.y >= V) ? PSTAT_DEV_BAD_LABEL
                                                                   : PSTAT_DEV_EMPTY_ROW);
                }
            }
        }
    }

    __device__ void tile(State& st, uint32_t taddr, int /*m*/, int n, int /*row*/) const {
        const int64_t j0 = (int64_t)n * BN;  // chunk-local column of the tile
        const uint64_t negM = f2_pack(-st.M, -st.M);
        const uint64_t l2e = f2_pack(kLog2e, kLog2e);
        const uint64_t nl2s = f2_pack(-st.log2S, -st.log2S);
        const float negw = -st.w;
        bool range = false;
        for (int p = 0; p < BN / 32; ++p) {
            const int64_t jp = j0 + p * 32;
            float v[32];
            tmem_ld32(taddr + p * 32, v);
            tmem_ld_wait();
            float g[32];
            if (st.live) {
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                    const uint64_t d = f2_add(f2_pack(v[i], v[i + 1]), negM);
                    float a0, a1;
                    f2_unpack(f2_fma(d, l2e, nl2s), a0, a1);
                    g[i] = negw * ex2_approx(a0);
                    g[i + 1] = negw * ex2_approx(a1);
                }
                const int64_t yl = st.y - c0 - jp;
                if (yl >= 0 && yl < 32) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (yl == i) g[i] = st.w + g[i];  // w (1 - p)
                }
                const int64_t vcol = c0 + jp;  // vocabulary index of column i is vcol + i
                if (vcol + 32 > V) {
                    for (int i = 0; i < 32; ++i)
                        if (vcol + i >= V) g[i] = 0.f;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) range |= fabsf(g[i]) > 65504.f;
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) g[i] = 0.f;
            }
            // G row segment: 32 fp16 = 4 x 16 bytes
            uint32_t h2[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const __half2 x = __floats2half2_rn(g[2 * i], g[2 * i + 1]);
                h2[i] = *reinterpret_cast<const uint32_t*>(&x);
            }
            uint4* gp = reinterpret_cast<uint4*>(G + st.t * ldg + jp);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                gp[i] = make_uint4(h2[4 * i], h2[4 * i + 1], h2[4 * i + 2], h2[4 * i + 3]);
            // Gt column: the 32 lanes of the warp hold 32 consecutive tokens
            __half* gtp = Gt + jp * ldgt + st.t;
#pragma unroll
            for (int i = 0; i < 32; ++i) gtp[(int64_t)i * ldgt] = __float2half_rn(g[i]);
        }
        if (range && dev_error) atomicOr(dev_error, PSTAT_DEV_RANGE);
    }

    __device__ void unit_end(State&, int, int, int) const {}
};

// Backward steps 2 and 3: out[row0 + r, c] += acc[r, c] for r < rows,
// c < cols, with 16-byte vector reductions (each element has exactly one
// writer per launch, so the result does not depend on timing).
struct AccumEpi {
    float* out;
    int64_t ld;
    int64_t row0;
    int64_t rows, cols;

    struct State {};

    __device__ void unit_begin(State&, int, int, int) const {}

    __device__ void tile(State&, uint32_t taddr, int m, int n, int row) const {
        const int64_t r = (int64_t)m * BM + row;
        const int64_t c0 = (int64_t)n * BN;
        for (int p = 0; p < BN / 32; ++p) {
            float v[32];
            tmem_ld32(taddr + p * 32, v);
            tmem_ld_wait();
            if (r >= rows) continue;
            float* dst = out + (row0 + r) * ld + c0 + p * 32;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                if (c0 + p * 32 + i + 4 <= cols)
                    red_add_v4(dst + i, v[i], v[i + 1], v[i + 2], v[i + 3]);
            }
        }
    }

    __device__ void unit_end(State&, int, int, int) const {}
};

// ---------------------------------------------------------------------------
// The GEMM kernel.
// ---------------------------------------------------------------------------
template <class Epi, bool kF16>
__global__ void __launch_bounds__(THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ Problems<Epi> P, int* __restrict__ dev_error) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem::bars);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* uq_full = drain + 1;
    uint64_t* uq_empty = uq_full + QD;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Smem::tmem_slot);
    volatile int* uq = reinterpret_cast<volatile int*>(smem + Smem::uq);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool dynamic = P.counter != nullptr;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        mbar_init(drain, 1);
        for (int q = 0; q < QD; ++q) {
            mbar_init(&uq_full[q], 1);   // the producer publishes a unit
            mbar_init(&uq_empty[q], 5);  // the MMA thread and the 4 epilogue warps took it
        }
        fence_mbar_init();
        prefetch_tensormap(&P.p[0].a);
        prefetch_tensormap(&P.p[0].b);
        if (P.total > P.n0) {
            prefetch_tensormap(&P.p[1].a);
            prefetch_tensormap(&P.p[1].b);
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    bool failed = false;

    // The i-th unit of this CTA for a consumer role: round robin, or popped
    // from the queue the producer fills.  -1 ends the loop; -2 is a timeout.
    auto consume_unit = [&](int64_t i, bool arrive) -> int64_t {
        if (!dynamic) {
            const int64_t u = (int64_t)blockIdx.x + i * gridDim.x;
            return u < P.total ? u : -1;
        }
        const int q = (int)(i % QD);
        if (!mbar_wait_bounded(&uq_full[q], (uint32_t)((i / QD) & 1), WAIT_NS)) return -2;
        const int64_t u = uq[q];
        if (arrive) mbar_arrive(&uq_empty[q]);
        return u;
    };

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint64_t pol_a = policy_evict_last();
            const uint64_t pol_b = policy_evict_first();
            uint32_t it = 0;
            for (int64_t i = 0; !failed; ++i) {
                int64_t u;
                if (dynamic) {
                    const int q = (int)(i % QD);
                    if (!mbar_wait_bounded(&uq_empty[q], (uint32_t)(((i / QD) & 1) ^ 1), WAIT_NS)) {
                        failed = true;
                        break;
                    }
                    u = atomicAdd(P.counter, 1);
                    if (u >= P.total) u = -1;
                    uq[q] = (int)u;
                    mbar_arrive(&uq_full[q]);
                } else {
                    u = (int64_t)blockIdx.x + i * gridDim.x;
                    if (u >= P.total) u = -1;
                }
                if (u < 0) break;
                const int w = u < P.n0 ? 0 : 1;
                const Problem<Epi>& pr = P.p[w];
                int m, un;
                unit_coords(pr.g, u - (w ? P.n0 : 0), m, un);
                const int nt = unit_tiles(pr.g, un);
                for (int j = 0; j < nt && !failed; ++j) {
                    const int n = un * pr.g.tiles_per_unit + j;
                    for (int kb = 0; kb < pr.g.k_blocks; ++kb, ++it) {
                        const int s = it % STAGES;
                        const uint32_t ph = (it / STAGES) & 1u;
                        if (!mbar_wait_bounded(&empty[s], ph ^ 1u, WAIT_NS)) {
                            failed = true;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                        tma_load_2d(smem + Smem::a + s * A_BYTES, &pr.a, kb * BK, m * BM,
                                    &full[s], pol_a);
                        tma_load_2d(smem + Smem::b + s * B_BYTES, &pr.b, kb * BK,
                                    pr.g.b_row0 + n * BN, &full[s], pol_b);
                    }
                }
            }
            // Every copy this thread issued must have landed before the CTA can
            // end (on the normal path they all have; after a timeout some may not).
            for (uint32_t k = 0; k < (uint32_t)STAGES && k < it; ++k) {
                const uint32_t i = it - 1 - k;
                if (!mbar_wait_bounded(&full[i % STAGES], (i / STAGES) & 1u, WAIT_NS))
                    failed = true;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = kF16 ? idesc_f16_f32(BM, BN) : idesc_bf16_f32(BM, BN);
            uint32_t it = 0, tc = 0;
            for (int64_t i = 0; !failed; ++i) {
                const int64_t u = consume_unit(i, true);
                if (u == -2) failed = true;
                if (u < 0) break;
                const int w = u < P.n0 ? 0 : 1;
                const GemmGeo& g = P.p[w].g;
                int m, un;
                unit_coords(g, u - (w ? P.n0 : 0), m, un);
                const int nt = unit_tiles(g, un);
                for (int j = 0; j < nt && !failed; ++j, ++tc) {
                    const uint32_t b = tc & 1u;
                    const uint32_t tph = (tc >> 1) & 1u;
                    if (!mbar_wait_bounded(&tempty[b], tph ^ 1u, WAIT_NS)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t d_tmem = tmem_base + b * BN;
                    for (int kb = 0; kb < g.k_blocks; ++kb, ++it) {
                        const int s = it % STAGES;
                        const uint32_t ph = (it / STAGES) & 1u;
                        if (!mbar_wait_bounded(&full[s], ph, WAIT_NS)) {
                            failed = true;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t a_addr = smem_u32(smem + Smem::a + s * A_BYTES);
                        const uint32_t b_addr = smem_u32(smem + Smem::b + s * B_BYTES);
#pragma unroll
                        for (int kk = 0; kk < BK / UK; ++kk) {
                            umma_bf16(d_tmem, sdesc_kmajor_sw128(a_addr + kk * UK * 2),
                                      sdesc_kmajor_sw128(b_addr + kk * UK * 2), idesc,
                                      (kb | kk) != 0);
                        }
                        umma_commit(&empty[s]);  // frees the stage once these MMAs finish
                    }
                    if (failed) break;
                    umma_commit(&tfull[b]);      // accumulator b is ready
                }
            }
            // All MMAs issued by this thread complete before tensor memory is freed.
            umma_commit(drain);
            if (!mbar_wait_bounded(drain, 0, WAIT_NS)) failed = true;
        }
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;  // TMEM lane quadrant of this warp
        const int row = q * 32 + lane;
        uint32_t tc = 0;
        typename Epi::State st;
        for (int64_t i = 0; !failed; ++i) {
            int64_t u = consume_unit(i, false);
            __syncwarp();
            if (dynamic && lane == 0 && u != -2) mbar_arrive(&uq_empty[i % QD]);
            u = __shfl_sync(0xFFFFFFFFu, u, 0);
            if (u == -2) failed = true;
            if (u < 0) break;
            const int w = u < P.n0 ? 0 : 1;
            const Problem<Epi>& pr = P.p[w];
            int m, un;
            unit_coords(pr.g, u - (w ? P.n0 : 0), m, un);
            const int nt = unit_tiles(pr.g, un);
            pr.epi.unit_begin(st, m, un, row);
            for (int j = 0; j < nt; ++j, ++tc) {
                const int n = un * pr.g.tiles_per_unit + j;
                const uint32_t b = tc & 1u;
                const uint32_t tph = (tc >> 1) & 1u;
                bool ok = mbar_wait_bounded(&tfull[b], tph, WAIT_NS);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) {
                    failed = true;
                    break;
                }
                tc_fence_after_sync();
                pr.epi.tile(st, tmem_base + ((uint32_t)(q * 32) << 16) + b * BN, m, n, row);
                // accumulator b may be overwritten from here on
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[b]);
            }
            if (failed) break;
            pr.epi.unit_end(st, m, un, row);
        }
    }

    if (failed && dev_error) atomicOr(dev_error, PSTAT_DEV_TIMEOUT);
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Transpose with conversion to fp16: dst[c, r] = fp16(src[r, c]) for r < rows,
// 0 for rows <= r < rows_pad; c < cols.  32 x 32 tiles through shared memory.
// Values beyond the fp16 range set PSTAT_DEV_RANGE.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
    transpose_bf16_to_f16(const uint16_t* __restrict__ src, int64_t rows, int64_t cols,
                          int64_t ld_src, __half* __restrict__ dst, int64_t ld_dst,
                          int64_t rows_pad, int* __restrict__ dev_error) {
    __shared__ float tile[32][33];
    const int64_t r0 = (int64_t)blockIdx.y * 32;
    const int64_t c0 = (int64_t)blockIdx.x * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    bool range = false;
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
        const int64_t r = r0 + ty + k, c = c0 + tx;
        float x = 0.f;
        if (r < rows && c < cols) x = __uint_as_float((uint32_t)src[r * ld_src + c] << 16);
        range |= fabsf(x) > 65504.f;
        tile[ty + k][tx] = x;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 32; k += 8) {
        const int64_t c = c0 + ty + k, r = r0 + tx;
        if (c < cols && r < rows_pad) dst[c * ld_dst + r] = __float2half_rn(tile[tx][ty + k]);
    }
    if (range && dev_error) atomicOr(dev_error, PSTAT_DEV_RANGE);
}

// ---- host side ------------------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major 16-bit matrix [rows, cols] (row stride ld elements) -> tensor map
// with box [box_rows, 64] and the 128-byte swizzle.
static bool make_map(CUtensorMap* map, bool f16, const void* ptr, int64_t rows, int64_t cols,
                     int64_t ld, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
              const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static GemmGeo geo(int64_t M, int64_t N, int64_t K, int tiles_per_unit, int64_t b_row0,
                   int m_group = M_GROUP) {
    GemmGeo g;
    g.m_group = m_group;
    g.m_tiles = (int)((M + BM - 1) / BM);
    g.n_tiles = (int)((N + BN - 1) / BN);
    g.k_blocks = (int)((K + BK - 1) / BK);
    g.tiles_per_unit = tiles_per_unit;
    g.units_per_m = (g.n_tiles + tiles_per_unit - 1) / tiles_per_unit;
    g.n_units = (int64_t)g.m_tiles * g.units_per_m;
    g.b_row0 = (int)b_row0;
    return g;
}

template <class Epi, bool kF16>
static cudaError_t launch_problems(const Problems<Epi>& P, int* dev_error, int sm_count,
                                   cudaStream_t st) {
    static std::atomic<bool> configured[64];
    int devi = 0;
    cudaGetDevice(&devi);
    if (devi >= 64 || !configured[devi].load()) {
        const cudaError_t e =
            cudaFuncSetAttribute(tc_gemm_kernel<Epi, kF16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        if (devi < 64) configured[devi].store(true);
    }
    if (P.total == 0) return cudaSuccess;
    const int64_t grid = P.total < sm_count ? P.total : sm_count;
    tc_gemm_kernel<Epi, kF16><<<(unsigned)grid, THREADS, SMEM_BYTES, st>>>(P, dev_error);
    return cudaGetLastError();
}

// One GEMM, static round-robin schedule.
template <class Epi, bool kF16>
static cudaError_t launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const GemmGeo& g,
                               const Epi& epi, int* dev_error, int sm_count, cudaStream_t st) {
    Problems<Epi> P;
    P.p[0].a = ma;
    P.p[0].b = mb;
    P.p[0].g = g;
    P.p[0].epi = epi;
    P.p[1] = P.p[0];
    P.n0 = g.n_units;
    P.total = g.n_units;
    P.counter = nullptr;
    return launch_problems<Epi, kF16>(P, dev_error, sm_count, st);
}

// Two GEMMs in one launch, units claimed through `counter` (zeroed before).
// The first problem should be the one with the longer units.
template <class Epi, bool kF16>
static cudaError_t launch_gemm_pair(const CUtensorMap& ma0, const CUtensorMap& mb0,
                                    const GemmGeo& g0, const Epi& e0, const CUtensorMap& ma1,
                                    const CUtensorMap& mb1, const GemmGeo& g1, const Epi& e1,
                                    int* counter, int* dev_error, int sm_count, cudaStream_t st) {
    Problems<Epi> P;
    P.p[0].a = ma0;
    P.p[0].b = mb0;
    P.p[0].g = g0;
    P.p[0].epi = e0;
    P.p[1].a = ma1;
    P.p[1].b = mb1;
    P.p[1].g = g1;
    P.p[1].epi = e1;
    P.n0 = g0.n_units;
    P.total = g0.n_units + g1.n_units;
    P.counter = counter;
    return launch_problems<Epi, kF16>(P, dev_error, sm_count, st);
}

static cudaError_t launch_transpose(const uint16_t* src, int64_t rows, int64_t cols,
                                    int64_t ld_src, __half* dst, int64_t ld_dst, int64_t rows_pad,
                                    int* dev_error, cudaStream_t st) {
    const dim3 grid((unsigned)((cols + 31) / 32), (unsigned)((rows_pad + 31) / 32));
    transpose_bf16_to_f16<<<grid, 256, 0, st>>>(src, rows, cols, ld_src, dst, ld_dst, rows_pad,
                                                 dev_error);
    return cudaGetLastError();
}

// A stream and events of one backward call: the W transposes run there, next
// to the GEMMs on the caller's stream.  Created per call and released at the
// end of it (destruction waits for nothing; the driver frees them once their
// work is done), so concurrent calls never share them.  Once forked from the
// caller's stream, the side stream is joined back into it when this object
// goes out of scope -- on every return path, errors included -- so nothing
// the call queued can outlive the caller's view of it.
struct SideStream {
    cudaStream_t s = nullptr, caller = nullptr;
    cudaEvent_t start = nullptr, hT = nullptr, done = nullptr, tr[2] = {}, acc[2] = {};
    bool ok = false, forked = false;
    SideStream() {
        ok = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) == cudaSuccess;
        for (cudaEvent_t* e : {&start, &hT, &done, &tr[0], &tr[1], &acc[0], &acc[1]})
            ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    }
    // The side stream's work starts after everything queued so far on `c`.
    bool fork(cudaStream_t c) {
        caller = c;
        forked = cudaEventRecord(start, c) == cudaSuccess &&
                 cudaStreamWaitEvent(s, start, 0) == cudaSuccess;
        return forked;
    }
    ~SideStream() {
        if (forked && cudaEventRecord(done, s) == cudaSuccess)
            cudaStreamWaitEvent(caller, done, 0);
        for (cudaEvent_t e : {start, hT, done, tr[0], tr[1], acc[0], acc[1]})
            if (e) cudaEventDestroy(e);
        if (s) cudaStreamDestroy(s);
    }
};

// ---- workspace layouts -------------------------------------------------------------
struct FwdWorkspace {
    size_t stats_off, target_off, total;
};
static FwdWorkspace fwd_layout(int64_t T, int64_t V) {
    const int64_t nc = (V + LM_CHUNK - 1) / LM_CHUNK;
    FwdWorkspace w;
    w.stats_off = 0;
    w.target_off = align_up((size_t)T * nc * kChunkRecordBytes, 256);
    w.total = align_up(w.target_off + (size_t)T * sizeof(float), 256);
    return w;
}

struct BwdWorkspace {
    int64_t Tp;  // T padded to whole M tiles
    size_t hT_off, Wt_off[2], G_off, Gt_off, ctr_off, total;
    int64_t n_chunks;  // vocabulary chunks of VC columns
};
static BwdWorkspace bwd_layout(int64_t T, int64_t V, int64_t d) {
    BwdWorkspace w;
    w.Tp = (T + BM - 1) / BM * BM;
    w.hT_off = 0;                                                 // [d, Tp] fp16
    w.Wt_off[0] = align_up(w.hT_off + (size_t)d * w.Tp * 2, 1024);  // [d, VC] fp16, two
    w.Wt_off[1] = align_up(w.Wt_off[0] + (size_t)d * VC * 2, 1024); // (chunks alternate)
    w.G_off = align_up(w.Wt_off[1] + (size_t)d * VC * 2, 1024);     // [Tp, VC] fp16
    w.Gt_off = align_up(w.G_off + (size_t)w.Tp * VC * 2, 1024);  // [VC, Tp] fp16
    w.ctr_off = align_up(w.Gt_off + (size_t)VC * w.Tp * 2, 1024);  // int[n_chunks]
    w.n_chunks = (V + VC - 1) / VC;
    w.total = align_up(w.ctr_off + (size_t)w.n_chunks * sizeof(int), 1024);
    return w;
}

static int check_lm_args(const void* hidden, const void* W, int64_t T, int64_t V, int64_t d) {
    if (T < 0 || V < 1 || d < BK || d % BK != 0 || d > (1 << 20)) return PSTAT_ERR_SHAPE;
    if (T > (int64_t)INT32_MAX / 2 || V > (int64_t)INT32_MAX / 2) return PSTAT_ERR_SHAPE;
    if (T == 0) return PSTAT_OK;
    if (!hidden || !W) return PSTAT_ERR_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(hidden) & 15u) || (reinterpret_cast<uintptr_t>(W) & 15u))
        return PSTAT_ERR_ALIGN;
    return PSTAT_OK;
}

}  // namespace lm
}  // namespace pstat

using namespace pstat;

extern "C" {

int pstat_lmhead_workspace_size(int64_t T, int64_t V, int64_t d, size_t* bytes) {
    if (!bytes) return PSTAT_ERR_NULLPTR;
    if (T < 0 || V < 1 || d < lm::BK || d % lm::BK != 0) return PSTAT_ERR_SHAPE;
    const size_t f = lm::fwd_layout(T, V).total;
    const size_t b = lm::bwd_layout(T, V, d).total;
    *bytes = f > b ? f : b;
    return PSTAT_OK;
}

int pstat_lmhead_fused(const void* hidden, const void* W, int64_t T, int64_t V, int64_t d,
                       const int64_t* labels, int64_t ignore_index, float* out_logprob,
                       float* out_entropy, float* out_rowstats, void* workspace,
                       size_t ws_bytes, int* dev_error, pstat_stream_t stream) {
    int rc = lm::check_lm_args(hidden, W, T, V, d);
    if (rc != PSTAT_OK || T == 0) return rc;
    const lm::FwdWorkspace wl = lm::fwd_layout(T, V);
    if (!workspace || ws_bytes < wl.total) return PSTAT_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return PSTAT_ERR_ALIGN;
    if ((labels && (reinterpret_cast<uintptr_t>(labels) & 7u)) ||
        (out_rowstats && (reinterpret_cast<uintptr_t>(out_rowstats) & 7u)))
        return PSTAT_ERR_ALIGN;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    ShardPlan plan;
    rc = make_plan(V, lm::LM_CHUNK, nullptr, 1, &plan);
    if (rc != PSTAT_OK) return rc;

    CUtensorMap map_h, map_w;
    if (!lm::make_map(&map_h, false, hidden, T, d, d, lm::BM) ||
        !lm::make_map(&map_w, false, W, V, d, d, lm::BN))
        return PSTAT_ERR_CUDA;
    char* ws = static_cast<char*>(workspace);
    lm::StatsEpi epi;
    epi.T = T;
    epi.V = V;
    epi.n_chunks = plan.n_chunks;
    epi.labels = labels;
    epi.ignore_index = ignore_index;
    epi.chunk_stats = reinterpret_cast<float4*>(ws + wl.stats_off);
    epi.target = reinterpret_cast<float*>(ws + wl.target_off);
    const lm::GemmGeo g = lm::geo(T, V, d, lm::STATS_TILES, 0);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (lm::launch_gemm<lm::StatsEpi, false>(map_h, map_w, g, epi, dev_error, dev.sm_count, st) !=
        cudaSuccess)
        return PSTAT_ERR_CUDA;
    if (launch_combine(epi.chunk_stats, plan, nullptr, PSTAT_BF16, T, V, V, labels, ignore_index,
                       epi.target, out_logprob, out_entropy, out_rowstats, dev_error,
                       st) != cudaSuccess)
        return PSTAT_ERR_CUDA;
    return PSTAT_OK;
}

int pstat_lmhead_backward(const void* hidden, const void* W, int64_t T, int64_t V, int64_t d,
                          const int64_t* labels, int64_t ignore_index, const float* weights,
                          const float* rowstats, float* dhidden, float* dW, void* workspace,
                          size_t ws_bytes, int* dev_error, pstat_stream_t stream) {
    int rc = lm::check_lm_args(hidden, W, T, V, d);
    if (rc != PSTAT_OK || T == 0) return rc;
    if (!rowstats || !dhidden || !dW) return PSTAT_ERR_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(dhidden) & 15u) || (reinterpret_cast<uintptr_t>(dW) & 15u) ||
        (reinterpret_cast<uintptr_t>(rowstats) & 7u) ||
        (labels && (reinterpret_cast<uintptr_t>(labels) & 7u)) ||
        (weights && (reinterpret_cast<uintptr_t>(weights) & 3u)))
        return PSTAT_ERR_ALIGN;
    const lm::BwdWorkspace wl = lm::bwd_layout(T, V, d);
    if (!workspace || ws_bytes < wl.total) return PSTAT_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 1023u) return PSTAT_ERR_ALIGN;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;

    char* ws = static_cast<char*>(workspace);
    __half* hT = reinterpret_cast<__half*>(ws + wl.hT_off);
    __half* Wt[2] = {reinterpret_cast<__half*>(ws + wl.Wt_off[0]),
                     reinterpret_cast<__half*>(ws + wl.Wt_off[1])};
    __half* G = reinterpret_cast<__half*>(ws + wl.G_off);
    __half* Gt = reinterpret_cast<__half*>(ws + wl.Gt_off);
    const int64_t Tp = wl.Tp;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    CUtensorMap map_h, map_w, map_G, map_Wt[2], map_Gt, map_hT;
    if (!lm::make_map(&map_h, false, hidden, T, d, d, lm::BM) ||
        !lm::make_map(&map_w, false, W, V, d, d, lm::BN) ||
        !lm::make_map(&map_G, true, G, Tp, lm::VC, lm::VC, lm::BM) ||
        !lm::make_map(&map_Wt[0], true, Wt[0], d, lm::VC, lm::VC, lm::BN) ||
        !lm::make_map(&map_Wt[1], true, Wt[1], d, lm::VC, lm::VC, lm::BN) ||
        !lm::make_map(&map_Gt, true, Gt, lm::VC, Tp, Tp, lm::BM) ||
        !lm::make_map(&map_hT, true, hT, d, Tp, Tp, lm::BN))
        return PSTAT_ERR_CUDA;

    lm::GradEpi ge;
    ge.T = T;
    ge.V = V;
    ge.labels = labels;
    ge.ignore_index = ignore_index;
    ge.weights = weights;
    ge.rowstats = reinterpret_cast<const float2*>(rowstats);
    ge.G = G;
    ge.ldg = lm::VC;
    ge.Gt = Gt;
    ge.ldgt = Tp;
    ge.dev_error = dev_error;

    const int64_t n_chunks = wl.n_chunks;
    int* ctr = reinterpret_cast<int*>(ws + wl.ctr_off);  // one unit counter per chunk
    if (cudaMemsetAsync(ctr, 0, (size_t)n_chunks * sizeof(int), st) != cudaSuccess)
        return PSTAT_ERR_CUDA;

    // The transposes (hidden once, W_c per chunk into alternating buffers) run
    // on a side stream: W_{c+1} is transposed while chunk c's GEMMs run, after
    // the GEMMs of chunk c-1 (the last reader of its buffer) are done.
    lm::SideStream x;
    if (!x.ok) return PSTAT_ERR_CUDA;
    auto transpose_w = [&](int64_t c) {
        const int64_t c0 = c * lm::VC;
        const int64_t vc = (V - c0) < lm::VC ? (V - c0) : lm::VC;
        // W_c^T (fp16; vocabulary columns past the chunk end as zeros)
        return lm::launch_transpose(static_cast<const uint16_t*>(W) + c0 * d, vc, d, d,
                                    Wt[c & 1], lm::VC, lm::VC, dev_error, x.s);
    };
    if (!x.fork(st)) return PSTAT_ERR_CUDA;
    // hidden^T once (fp16, tokens padded to Tp with zeros)
    if (lm::launch_transpose(static_cast<const uint16_t*>(hidden), T, d, d, hT, Tp, Tp, dev_error,
                             x.s) != cudaSuccess ||
        cudaEventRecord(x.hT, x.s) != cudaSuccess || transpose_w(0) != cudaSuccess ||
        cudaEventRecord(x.tr[0], x.s) != cudaSuccess)
        return PSTAT_ERR_CUDA;

    for (int64_t c = 0; c < n_chunks; ++c) {
        const int64_t c0 = c * lm::VC;
        const int64_t vc = (V - c0) < lm::VC ? (V - c0) : lm::VC;
        const int b = (int)(c & 1);
        if (c + 1 < n_chunks) {
            if (c >= 1 && cudaStreamWaitEvent(x.s, x.acc[b ^ 1], 0) != cudaSuccess)
                return PSTAT_ERR_CUDA;
            if (transpose_w(c + 1) != cudaSuccess ||
                cudaEventRecord(x.tr[b ^ 1], x.s) != cudaSuccess)
                return PSTAT_ERR_CUDA;
        }
        // 1. recompute the chunk's logits -> G, Gt
        ge.c0 = c0;
        const lm::GemmGeo g1 = lm::geo(Tp, vc, d, 1, c0);
        if (lm::launch_gemm<lm::GradEpi, false>(map_h, map_w, g1, ge, dev_error, dev.sm_count,
                                                st) != cudaSuccess)
            return PSTAT_ERR_CUDA;
        if (cudaStreamWaitEvent(st, x.tr[b], 0) != cudaSuccess ||
            (c == 0 && cudaStreamWaitEvent(st, x.hT, 0) != cudaSuccess))
            return PSTAT_ERR_CUDA;
        // 2. dhidden += G W_c  and  3. dW[c0 : c0 + vc] += Gt hidden, in one
        // launch: CTAs claim units of both GEMMs (the longer-K one first)
        // from this chunk's counter, so neither leaves a partial last wave.
        lm::AccumEpi e2;
        e2.out = dhidden;
        e2.ld = d;
        e2.row0 = 0;
        e2.rows = T;
        e2.cols = d;
        const lm::GemmGeo g2 = lm::geo(T, d, vc, 1, 0, lm::ACC_M_GROUP);
        lm::AccumEpi e3;
        e3.out = dW;
        e3.ld = d;
        e3.row0 = c0;
        e3.rows = vc;
        e3.cols = d;
        const lm::GemmGeo g3 = lm::geo(vc, d, Tp, 1, 0, lm::ACC_M_GROUP);
        const cudaError_t e =
            g3.k_blocks >= g2.k_blocks
                ? lm::launch_gemm_pair<lm::AccumEpi, true>(map_Gt, map_hT, g3, e3, map_G,
                                                           map_Wt[b], g2, e2, ctr + c, dev_error,
                                                           dev.sm_count, st)
                : lm::launch_gemm_pair<lm::AccumEpi, true>(map_G, map_Wt[b], g2, e2, map_Gt,
                                                           map_hT, g3, e3, ctr + c, dev_error,
                                                           dev.sm_count, st);
        if (e != cudaSuccess || cudaEventRecord(x.acc[b], st) != cudaSuccess)
            return PSTAT_ERR_CUDA;
    }
    // x joins the side stream back into st as it goes out of scope
    return PSTAT_OK;
}

}  // extern "C"
