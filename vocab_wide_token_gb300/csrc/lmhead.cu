// lmhead.cu -- fused lm_head on the 5th-generation tensor cores.
//
// Forward: logits z = hidden W^T are produced tile by tile (128 tokens x 256
// vocabulary rows, K = d in steps of 64) by tcgen05.mma into tensor memory
// and folded straight into the per-(token, 4096-column chunk) statistics
// (m, s, u) that the unfused path also produces; the logits never reach
// global memory.  The fixed-order combine kernel then gives logprob, entropy
// and (M, ln S).
//
// Backward (the chunked lm_head of TRL PR #6949 "ZeroSyncGRPOTrainer": GEMMs
// in a 16-bit dtype, accumulation in fp32 buffers).  With g = w q, where
// q = onehot(y) - e^(z - M - ln S) lies in [-1, 1] and depends on the row
// alone:
//   0. once per call, W -> W16 = fp16(W) [V, d] and hidden -> h' =
//      fp16(w_t hidden_t) [T, d] (one memory-bound launch);
//   per 32768-column vocabulary chunk c:
//   1. recompute the chunk's logits tile by tile and turn them on chip into
//      G = fp16(-2^15 q) [T, Vc] (row-major; the sign is the accumulation's);
//   2. dhidden += (-w_t 2^-15) (G W16_c)  A = G (K-major), B = W16_c read in
//                                          place (MN-major);
//   3. dW[c]   += -2^-15 (G^T h')         A = G read in place (MN-major),
//                                          B = h' (MN-major).
// Why the scale: at V = 151,936 nearly every softmax probability is below
// 2^-14, where fp16 numbers are subnormal and lose relative precision; 2^15 q
// keeps every |q| >= 2^-29 normal (and |2^15 q| <= 2^15 < 65504), so each
// element carries one fp16 rounding (2^-12 relative) whatever its size.  The
// weight is applied outside G (per output row of dhidden, folded into h' for
// dW), so a token's G row -- and its dhidden row -- does not depend on the
// other tokens of the batch.  fp16 (11-bit significand) rather than bf16
// (8 bits, about 2e-3 relative) keeps dhidden and dW within 1e-3.  W converts
// to fp16 exactly for 2^-14 <= |x| <= 65504; values above, and w hidden above
// 65504, flag PSTAT_DEV_RANGE.
//
// One warp-specialised persistent GEMM kernel serves every step (192
// threads, one CTA per SM):
//   warp 0     TMA producer: 2-D tiled loads of A (128 x 64) and B (256 x 64)
//              k-blocks into a 4-stage shared-memory ring (128-byte swizzle);
//              an operand stored with its M or N index contiguous (MN-major)
//              arrives as 64 x 64 boxes and is read in place
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
// Statistics chunk of the fused forward: 2048 vocabulary columns (8 tiles),
// folded in ascending tile order by one CTA.  Half the 4096 of the logits
// path: at V = 151,936 a 16-tile unit leaves some SMs 32 units (512 tiles)
// against an average of 500; 8-tile units cap that at 504.
constexpr int LM_CHUNK = 2048;
constexpr int STATS_TILES = LM_CHUNK / BN;
// Backward vocabulary chunk (columns staged as G).  Wider chunks give each
// accumulation launch more units, so its last partial wave weighs less, and
// fewer launches: at T = 16384, 8192 columns took 39.2-39.4 ms per backward,
// 16384 columns 38.1-38.6 ms, and 32768 columns 0.7% less again (same-box
// A/B, three pairs).  The width is a constant: it fixes the order in which a
// dhidden element accumulates the chunks.
constexpr int VC = 32768;
// G holds -2^15 q, q = onehot(y) - p in [-1, 1]: no |q| >= 2^-29 is subnormal
// in fp16 and |2^15 q| <= 32768 < 65504.  The accumulation GEMMs multiply by
// GRAD_UNSCALE = -2^-15 (exact), which restores q and its sign.
constexpr float GRAD_SCALE = 32768.f;
constexpr float GRAD_UNSCALE = -1.f / 32768.f;
constexpr int M_GROUP = 32;        // M tiles sharing the L2-resident slice of A
// The accumulation GEMMs run with 256-row tiles (TileCfg<true>): measured on
// their shapes (8192 x 4096 x 16384 and 16384 x 4096 x 8192), 3% and 11%
// faster than 128-row tiles, bit-identical.  Groups of 8 such tiles (2048
// rows of A, as 16 tiles of 128 rows before) were within 1-2% of 4 and 16 and
// ahead of 32.
constexpr bool ACC_WIDE = true;
// Tile configuration of the forward statistics GEMM and of the backward's
// recompute GEMM.  256-row tiles gave the same bits and no measurable gain
// there (forward 11.73-11.82 against 11.58-11.89 ms, backward 39.2-40.0
// against 39.7-39.9 ms, same box): their epilogues are heavier and their K
// (= d) shorter, so the undoubled accumulator costs what the operand traffic
// saves.
constexpr bool FWD_WIDE = false;
constexpr bool GRAD_WIDE = false;
constexpr int ACC_M_GROUP = 8;
constexpr uint32_t B_BYTES = BN * BK * 2;   // 32 KB
constexpr uint32_t TMEM_COLS = 2 * BN;      // two 128 x 256 fp32 accumulators
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr int QD = 4;  // depth of the claimed-unit queue (dynamic scheduling)

// Tile configuration of one GEMM kernel instantiation.
//   kWide = false: 128 x 256 output tiles, 4 pipeline stages of 48 KB, the two
//     TMEM accumulators double-buffer consecutive tiles, 4 epilogue warps.
//   kWide = true: 256 x 256 output tiles computed as two M = 128 MMAs that
//     share each B k-block, 3 stages of 64 KB, both accumulators hold one
//     tile (no double buffer: the next tile waits for the drain), 8 epilogue
//     warps (one per TMEM lane quadrant and accumulator).  Per k-block an SM
//     loads 64 KB for 2 x 128 x 256 x 64 MMA work instead of 48 KB for half
//     of it: a third less L2-to-SM operand traffic per flop, for GEMMs whose
//     K is long enough to hide the undoubled drain.
template <bool kWide>
struct TileCfg {
    static constexpr int TM = kWide ? 256 : 128;  // output rows per tile
    static constexpr int HALVES = TM / BM;        // M = 128 MMAs per k-step
    static constexpr int STAGES = kWide ? 3 : 4;
    static constexpr uint32_t A_BYTES = TM * BK * 2;
    static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int EPI_WARPS = 4 * HALVES;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int ACC_BUFS = kWide ? 1 : 2;  // tiles in flight in tensor memory
    // Offsets inside the 1024-byte aligned dynamic shared memory block.
    static constexpr uint32_t a = 0;
    static constexpr uint32_t b = a + STAGES * A_BYTES;
    static constexpr uint32_t bars = b + STAGES * B_BYTES;
    // full[STAGES], empty[STAGES], tfull[2], tempty[2], drain, uq_full[QD], uq_empty[QD]
    static constexpr uint32_t n_bars = 2 * STAGES + 4 + 1 + 2 * QD;
    static constexpr uint32_t tmem_slot = bars + n_bars * 8;
    static constexpr uint32_t uq = tmem_slot + 16;  // int[QD]: claimed unit ids
    static constexpr uint32_t total = uq + QD * 4;
    static constexpr size_t SMEM_BYTES = total + 1024;  // + alignment slack
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
    static_assert(a % 1024 == 0 && b % 1024 == 0 && A_BYTES % 1024 == 0,
                  "stages must keep the 1 KB alignment of the 128-byte swizzle");
};

struct GemmGeo {
    int m_tiles, n_tiles, k_blocks;
    int tiles_per_unit;   // consecutive N tiles one CTA processes in order
    int units_per_m;      // ceil(n_tiles / tiles_per_unit)
    int64_t n_units;      // m_tiles * units_per_m
    int b_n0;             // B's N coordinate of N tile 0 (tensor-map coordinate)
    int b_k0;             // B's K coordinate of k-block 0
    int m_group;          // M tiles per group: units run M-fastest within a group
};

// Operand layouts, a compile-time parameter of the GEMM kernel (so the
// K-major-only instantiations carry no layout code): bit 0 / 1 = problem 0's
// A / B is MN-major, bit 2 / 3 = problem 1's.  K-major: a 2-D tensor map whose
// inner coordinate is K; one box is [rows of M or N] x 64 K.  MN-major: a 4-D
// tensor map {64 MN, 8 K rows, MN / 64, K / 8} (make_map_mn4d) and one box
// {64, 8, tile / 64, 8} per stage, which lays the 1 KB swizzle atoms out
// MN-first inside each 8-row K group: atom (K group g, MN block i) at
// (g * tile / 64 + i) KB.  Measured on a 8192 x 4096 x 16384 fp16 GEMM, both
// operands MN-major in this order run within 2% of both K-major, while one
// 64 x 64 box per MN block (atoms 8 KB apart) ran 14% slower.
__host__ __device__ constexpr uint32_t layout_bits(int a0, int b0, int a1, int b1) {
    return (uint32_t)(a0 != 0) | ((uint32_t)(b0 != 0) << 1) | ((uint32_t)(a1 != 0) << 2) |
           ((uint32_t)(b1 != 0) << 3);
}
template <uint32_t kLayout>
__device__ __forceinline__ bool a_mn_of(int w) {
    return ((kLayout >> (2 * w)) & 1u) != 0;
}
template <uint32_t kLayout>
__device__ __forceinline__ bool b_mn_of(int w) {
    return ((kLayout >> (2 * w + 1)) & 1u) != 0;
}

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
// What an epilogue warp hands to its policy besides the accumulator: the
// problem's output tensor map (for policies that store tiles with TMA), the
// warp's staging area in shared memory (Epi::kStageBytes) and which half of
// it is next.
struct EpiCtx {
    const CUtensorMap* cmap;
    uint8_t* stage;
    uint32_t next;
};

template <class Epi>
struct Problem {
    CUtensorMap a, b;
    CUtensorMap c;  // output map of the epilogue, where it stores tiles by TMA
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
// Operand-major bits of the instruction descriptor: bit 15 for A, bit 16 for
// B; set = MN-major.
__host__ __device__ constexpr uint32_t idesc_major(int a_mn, int b_mn) {
    return ((uint32_t)(a_mn != 0) << 15) | ((uint32_t)(b_mn != 0) << 16);
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

    static constexpr uint32_t kStageBytes = 0;
    static constexpr bool kBEvictFirst = true;  // each W k-block is read in one wave

    __device__ void tile(State& st, uint32_t taddr, int /*m*/, int n, int /*row*/,
                         EpiCtx&) const {
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

    __device__ void finish(EpiCtx&, int) const {}
};

// Backward step 1: the recomputed logits tile becomes the scaled gradient
// tile G = 2^15 (e^(z - M - ln S) - onehot(y)) = -2^15 q, stored as fp16 by
// TMA through the problem's output map (G [rows, chunk width], row-major).  The scale is folded into the exponent,
// 2^15 p = 2^((z - M) log2 e + 15 - log2 S): per pair of elements one packed
// subtract, one packed FMA and two exponentials, and the sign of q is left to
// the accumulation GEMMs' per-row factor.  Rows past T, columns past V,
// ignored rows and zero-weight rows are written as +0 (the weight itself is
// applied by the accumulation GEMMs).
struct GradEpi {
    int64_t T, V;
    int64_t c0;            // first vocabulary column of this chunk
    const int64_t* labels;
    int64_t ignore_index;
    const float* weights;
    const float2* rowstats;
    int* dev_error;

    struct State {
        int64_t t, y;
        bool live;
        float M, c15;  // c15 = 15 - log2 S
    };

    __device__ void unit_begin(State& st, int m, int /*un*/, int row) const {
        st.t = (int64_t)m * BM + row;
        st.live = false;
        st.y = ignore_index;
        st.M = 0.f;
        st.c15 = 0.f;
        if (st.t < T) {
            st.y = labels ? labels[st.t] : ignore_index;
            const float w = weights ? weights[st.t] : 1.f;
            if (st.y != ignore_index && w != 0.f) {
                const float2 rs = rowstats[st.t];
                st.M = rs.x;
                st.c15 = 15.f - rs.y * kLog2e;
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

    // Each epilogue warp owns 32 rows of the tile.  Their G values go out 64
    // columns at a time: written into one half of the warp's staging area
    // (32 rows x 128 bytes, the 128-byte swizzle: 16-byte chunk c of row r at
    // chunk c ^ (r & 7)), then stored by one lane with a TMA tensor store that
    // writes whole 128-byte lines.  A lane writing its own row straight to
    // global memory would put 32 rows' half sectors in every store.
    static constexpr uint32_t kHalfBytes = 32 * 128;
    static constexpr uint32_t kStageBytes = 2 * kHalfBytes;
    static constexpr bool kBEvictFirst = true;  // each W k-block is read in one wave

    __device__ void tile(State& st, uint32_t taddr, int /*m*/, int n, int row,
                         EpiCtx& ctx) const {
        const int lane = row & 31;
        const int64_t j0 = (int64_t)n * BN;  // chunk-local column of the tile
        const int t0 = (int)(st.t - lane);   // first row of this warp
        const uint64_t negM = f2_pack(-st.M, -st.M);
        const uint64_t l2e = f2_pack(kLog2e, kLog2e);
        const uint64_t c15 = f2_pack(st.c15, st.c15);
        for (int pp = 0; pp < BN / 64; ++pp) {
            uint8_t* half = ctx.stage + (ctx.next & 1u) * kHalfBytes;
            ++ctx.next;
            // the store that last read this half (two stores ago) is done reading
            if (lane == 0) bulk_wait_group_read<1>();
            __syncwarp();
            for (int hh = 0; hh < 2; ++hh) {
                const int p = 2 * pp + hh;
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
                        f2_unpack(f2_fma(d, l2e, c15), a0, a1);
                        g[i] = ex2_approx(a0);      // 2^15 p
                        g[i + 1] = ex2_approx(a1);
                    }
                    const int64_t yl = st.y - c0 - jp;
                    if (yl >= 0 && yl < 32) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (yl == i) g[i] = g[i] - GRAD_SCALE;  // 2^15 (p - 1)
                    }
                    const int64_t vcol = c0 + jp;  // vocabulary index of column i is vcol + i
                    if (vcol + 32 > V) {
                        for (int i = 0; i < 32; ++i)
                            if (vcol + i >= V) g[i] = 0.f;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) g[i] = 0.f;
                }
                uint32_t h2[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const __half2 x = __floats2half2_rn(g[2 * i], g[2 * i + 1]);
                    h2[i] = *reinterpret_cast<const uint32_t*>(&x);
                }
                // 32 fp16 = 4 chunks of this row, chunks 4 hh .. 4 hh + 3
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = (4 * hh + i) ^ (lane & 7);
                    *reinterpret_cast<uint4*>(half + lane * 128 + c * 16) =
                        make_uint4(h2[4 * i], h2[4 * i + 1], h2[4 * i + 2], h2[4 * i + 3]);
                }
            }
            fence_proxy_async_smem();  // the writes above precede the store's reads
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(ctx.cmap, (int)(j0 + pp * 64), t0, half);
                bulk_commit_group();
            }
        }
    }

    __device__ void unit_end(State&, int, int, int) const {}

    // Every store this warp issued has completed before the CTA ends.
    __device__ void finish(EpiCtx&, int row) const {
        if ((row & 31) == 0) bulk_wait_group<0>();
        __syncwarp();
    }
};

// Backward steps 2 and 3: out[row0 + r, c] += f_r acc[r, c] for r < rows,
// c < cols, with 16-byte vector reductions (each element has exactly one
// writer per launch, so the result does not depend on timing).  The factor
// is f_r = row_scale[r] * scale (row_scale may be NULL: f_r = scale); rows
// with f_r == 0 are skipped.
struct AccumEpi {
    float* out;
    int64_t ld;
    int64_t row0;
    int64_t rows, cols;
    const float* row_scale;
    float scale;

    struct State {};

    __device__ void unit_begin(State&, int, int, int) const {}

    static constexpr uint32_t kStageBytes = 0;
    // A B slice (K long, 8-16 MB) serves the 9-10 M tiles of a wave, whose CTAs
    // reach each k-block at different times: left at normal L2 priority it
    // stays for the later ones.
    static constexpr bool kBEvictFirst = false;

    __device__ void tile(State&, uint32_t taddr, int m, int n, int row, EpiCtx&) const {
        const int64_t r = (int64_t)m * BM + row;
        const int64_t c0 = (int64_t)n * BN;
        float f = 0.f;
        if (r < rows) f = row_scale ? row_scale[r] * scale : scale;
        for (int p = 0; p < BN / 32; ++p) {
            float v[32];
            tmem_ld32(taddr + p * 32, v);
            tmem_ld_wait();
            if (f == 0.f) continue;
            float* dst = out + (row0 + r) * ld + c0 + p * 32;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                if (c0 + p * 32 + i + 4 <= cols)
                    red_add_v4(dst + i, f * v[i], f * v[i + 1], f * v[i + 2], f * v[i + 3]);
            }
        }
    }

    __device__ void unit_end(State&, int, int, int) const {}

    __device__ void finish(EpiCtx&, int) const {}
};

// ---------------------------------------------------------------------------
// The GEMM kernel.
// ---------------------------------------------------------------------------
// Shared memory of a GEMM kernel instantiation: the tile configuration's
// layout, then (1 KB aligned) each epilogue warp's staging area.
template <bool kWide>
__host__ __device__ constexpr uint32_t stage_offset() {
    return (TileCfg<kWide>::total + 1023u) & ~1023u;
}
template <class Epi, bool kWide>
__host__ __device__ constexpr size_t gemm_smem_bytes() {
    return stage_offset<kWide>() + (size_t)TileCfg<kWide>::EPI_WARPS * Epi::kStageBytes +
           1024;  // + alignment slack
}

template <class Epi, bool kF16, uint32_t kLayout, bool kWide>
__global__ void __launch_bounds__(TileCfg<kWide>::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ Problems<Epi> P, int* __restrict__ dev_error) {
    using C = TileCfg<kWide>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::bars);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::STAGES;
    uint64_t* tfull = bars + 2 * C::STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint64_t* uq_full = drain + 1;
    uint64_t* uq_empty = uq_full + QD;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::tmem_slot);
    volatile int* uq = reinterpret_cast<volatile int*>(smem + C::uq);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool dynamic = P.counter != nullptr;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], C::EPI_WARPS);
        }
        mbar_init(drain, 1);
        for (int q = 0; q < QD; ++q) {
            mbar_init(&uq_full[q], 1);  // the producer publishes a unit
            // the MMA thread and every epilogue warp took it
            mbar_init(&uq_empty[q], 1 + C::EPI_WARPS);
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
            const uint64_t pol_b = Epi::kBEvictFirst ? policy_evict_first() : policy_evict_normal();
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
                        const int s = it % C::STAGES;
                        const uint32_t ph = (it / C::STAGES) & 1u;
                        if (!mbar_wait_bounded(&empty[s], ph ^ 1u, WAIT_NS)) {
                            failed = true;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
                        uint8_t* a_dst = smem + C::a + s * C::A_BYTES;
                        uint8_t* b_dst = smem + C::b + s * B_BYTES;
                        if (!a_mn_of<kLayout>(w))
                            tma_load_2d(a_dst, &pr.a, kb * BK, m * C::TM, &full[s], pol_a);
                        else
                            tma_load_4d(a_dst, &pr.a, 0, 0, m * (C::TM / 64), kb * (BK / 8),
                                        &full[s], pol_a);
                        const int bk = pr.g.b_k0 + kb * BK;
                        if (!b_mn_of<kLayout>(w))
                            tma_load_2d(b_dst, &pr.b, bk, pr.g.b_n0 + n * BN, &full[s], pol_b);
                        else
                            tma_load_4d(b_dst, &pr.b, 0, 0, (pr.g.b_n0 + n * BN) / 64, bk / 8,
                                        &full[s], pol_b);
                    }
                }
            }
            // Every copy this thread issued must have landed before the CTA can
            // end (on the normal path they all have; after a timeout some may not).
            for (uint32_t k = 0; k < (uint32_t)C::STAGES && k < it; ++k) {
                const uint32_t i = it - 1 - k;
                if (!mbar_wait_bounded(&full[i % C::STAGES], (i / C::STAGES) & 1u, WAIT_NS))
                    failed = true;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc0 = kF16 ? idesc_f16_f32(BM, BN) : idesc_bf16_f32(BM, BN);
            // K-major: the K step moves 32 bytes along the swizzled row and the
            // second 128-row half starts 128 rows x 128 bytes on.  MN-major
            // (atoms MN-first): the next MN block is 1 KB on, the next 8-row K
            // group (tile / 64) KB on, a K step of 16 rows spans two groups,
            // and the second half starts two MN blocks on.
            constexpr uint32_t a_kg = (C::TM / 64) * 1024, b_kg = (BN / 64) * 1024;
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
                const bool a_mn = a_mn_of<kLayout>(w), b_mn = b_mn_of<kLayout>(w);
                const uint32_t idesc = idesc0 | idesc_major(a_mn, b_mn);
                for (int j = 0; j < nt && !failed; ++j, ++tc) {
                    const uint32_t b = tc % C::ACC_BUFS;
                    const uint32_t tph = (tc / C::ACC_BUFS) & 1u;
                    if (!mbar_wait_bounded(&tempty[b], tph ^ 1u, WAIT_NS)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after_sync();
                    for (int kb = 0; kb < g.k_blocks; ++kb, ++it) {
                        const int s = it % C::STAGES;
                        const uint32_t ph = (it / C::STAGES) & 1u;
                        if (!mbar_wait_bounded(&full[s], ph, WAIT_NS)) {
                            failed = true;
                            break;
                        }
                        tc_fence_after_sync();
                        const uint32_t a_addr = smem_u32(smem + C::a + s * C::A_BYTES);
                        const uint32_t b_addr = smem_u32(smem + C::b + s * B_BYTES);
#pragma unroll
                        for (int kk = 0; kk < BK / UK; ++kk) {
                            const uint64_t bd =
                                b_mn ? sdesc_mnmajor_sw128(b_addr + kk * 2 * b_kg, 1024, b_kg)
                                     : sdesc_kmajor_sw128(b_addr + kk * UK * 2);
#pragma unroll
                            for (int h = 0; h < C::HALVES; ++h) {
                                const uint64_t ad =
                                    a_mn ? sdesc_mnmajor_sw128(
                                               a_addr + kk * 2 * a_kg + h * 2048, 1024, a_kg)
                                         : sdesc_kmajor_sw128(a_addr + h * (BM * 128) +
                                                              kk * UK * 2);
                                const uint32_t d_tmem = tmem_base + (kWide ? h : b) * BN;
                                umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0);
                            }
                        }
                        umma_commit(&empty[s]);  // frees the stage once these MMAs finish
                    }
                    if (failed) break;
                    umma_commit(&tfull[b]);      // the tile's accumulators are ready
                }
            }
            // All MMAs issued by this thread complete before tensor memory is freed.
            umma_commit(drain);
            if (!mbar_wait_bounded(drain, 0, WAIT_NS)) failed = true;
        }
    } else {
        // ---------------- epilogue ----------------
        const int q = warp & 3;                   // TMEM lane quadrant of this warp
        const int h = kWide ? (warp - 2) / 4 : 0;  // which 128-row half (wide tiles)
        const int row = q * 32 + lane;
        uint32_t tc = 0;
        typename Epi::State st;
        EpiCtx ctx;
        ctx.cmap = nullptr;
        ctx.stage = smem + stage_offset<kWide>() + (uint32_t)(warp - 2) * Epi::kStageBytes;
        ctx.next = 0;
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
            const int m128 = m * C::HALVES + h;  // this warp's 128-row tile
            ctx.cmap = &pr.c;
            pr.epi.unit_begin(st, m128, un, row);
            for (int j = 0; j < nt; ++j, ++tc) {
                const int n = un * pr.g.tiles_per_unit + j;
                const uint32_t b = tc % C::ACC_BUFS;
                const uint32_t tph = (tc / C::ACC_BUFS) & 1u;
                bool ok = mbar_wait_bounded(&tfull[b], tph, WAIT_NS);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) {
                    failed = true;
                    break;
                }
                tc_fence_after_sync();
                pr.epi.tile(st, tmem_base + ((uint32_t)(q * 32) << 16) + (kWide ? h : b) * BN,
                            m128, n, row, ctx);
                // the accumulator may be overwritten once every epilogue warp arrived
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[b]);
            }
            if (failed) break;
            pr.epi.unit_end(st, m128, un, row);
        }
        P.p[0].epi.finish(ctx, row);
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
// Backward step 0: W16 = fp16(W) [Vp, d] and h' = fp16(w_t hidden_t) [Tp, d]
// (rows V <= v < Vp and T <= t < Tp as +0; weights NULL = 1), 8 elements per
// thread and iteration, 16-byte loads and stores.  Values beyond the fp16
// range set PSTAT_DEV_RANGE.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 f16x8(const float (&x)[8], bool& range) {
    uint32_t h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        range |= fabsf(x[2 * i]) > 65504.f || fabsf(x[2 * i + 1]) > 65504.f;
        const __half2 v = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
        h[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
    return make_uint4(h[0], h[1], h[2], h[3]);
}

__global__ void __launch_bounds__(256)
    to_fp16_kernel(const uint16_t* __restrict__ W, int64_t nW8, int64_t nWp8,
                   __half* __restrict__ W16, const uint16_t* __restrict__ hidden,
                   const float* __restrict__ weights, int64_t T, int64_t Tp, int64_t d8,
                   __half* __restrict__ h16, int* __restrict__ dev_error) {
    bool range = false;
    const int64_t total = nWp8 + Tp * d8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        float x[8];
        uint4 out;
        if (i >= nW8 && i < nWp8) {
            reinterpret_cast<uint4*>(W16)[i] = make_uint4(0u, 0u, 0u, 0u);
        } else if (i < nW8) {
            const uint4 q = __ldcs(reinterpret_cast<const uint4*>(W) + i);
            const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[2 * k] = bf2_lo(w4[k]);
                x[2 * k + 1] = bf2_hi(w4[k]);
            }
            out = f16x8(x, range);
            reinterpret_cast<uint4*>(W16)[i] = out;
        } else {
            const int64_t j = i - nWp8;
            const int64_t t = j / d8;
            if (t < T) {
                const float wt = weights ? weights[t] : 1.f;
                const uint4 q = __ldcs(reinterpret_cast<const uint4*>(hidden) + j);
                const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    x[2 * k] = wt * bf2_lo(w4[k]);
                    x[2 * k + 1] = wt * bf2_hi(w4[k]);
                }
                out = f16x8(x, range);
            } else {
                out = make_uint4(0u, 0u, 0u, 0u);
            }
            reinterpret_cast<uint4*>(h16)[j] = out;
        }
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

// M x N output, K-long reduction; B's N and K tensor-map coordinates start
// at b_n0 and b_k0.
// MN-major 16-bit matrix [K rows, MN cols] (row stride ld elements; MN a
// multiple of 64, K a multiple of 8) -> 4-D tensor map {64, 8, MN / 64, K / 8}
// whose box {64, 8, tile_mn / 64, BK / 8} lays the swizzle atoms out MN-first
// within each 8-row K group.
static bool make_map_mn4d(CUtensorMap* map, const void* ptr, int64_t krows, int64_t mn,
                          int64_t ld, int tile_mn) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || mn % 64 != 0 || krows % 8 != 0) return false;
    const cuuint64_t dims[4] = {64, 8, (cuuint64_t)(mn / 64), (cuuint64_t)(krows / 8)};
    const cuuint64_t strides[3] = {(cuuint64_t)ld * 2, 128, (cuuint64_t)ld * 2 * 8};
    const cuuint32_t box[4] = {64, 8, (cuuint32_t)(tile_mn / 64), (cuuint32_t)(BK / 8)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static GemmGeo geo(int64_t M, int64_t N, int64_t K, int tiles_per_unit, int64_t b_n0,
                   int m_group = M_GROUP, int64_t b_k0 = 0, int tile_m = BM) {
    GemmGeo g;
    g.m_group = m_group;
    g.m_tiles = (int)((M + tile_m - 1) / tile_m);
    g.n_tiles = (int)((N + BN - 1) / BN);
    g.k_blocks = (int)((K + BK - 1) / BK);
    g.tiles_per_unit = tiles_per_unit;
    g.units_per_m = (g.n_tiles + tiles_per_unit - 1) / tiles_per_unit;
    g.n_units = (int64_t)g.m_tiles * g.units_per_m;
    g.b_n0 = (int)b_n0;
    g.b_k0 = (int)b_k0;
    return g;
}

template <class Epi, bool kF16, uint32_t kLayout, bool kWide>
static cudaError_t launch_problems(const Problems<Epi>& P, int* dev_error, int sm_count,
                                   cudaStream_t st) {
    using C = TileCfg<kWide>;
    constexpr size_t smem = gemm_smem_bytes<Epi, kWide>();
    static_assert(smem <= 227 * 1024, "shared memory per CTA");
    static ContextSeen configured;
    const cudaError_t e = ensure_smem_optin(
        reinterpret_cast<const void*>(tc_gemm_kernel<Epi, kF16, kLayout, kWide>), (int)smem,
        configured);
    if (e != cudaSuccess) return e;
    if (P.total == 0) return cudaSuccess;
    const int64_t grid = P.total < sm_count ? P.total : sm_count;
    tc_gemm_kernel<Epi, kF16, kLayout, kWide>
        <<<(unsigned)grid, C::THREADS, smem, st>>>(P, dev_error);
    return cudaGetLastError();
}

// One GEMM, static round-robin schedule, both operands K-major, tile
// configuration kWide (the geometry's M tiles must be TileCfg<kWide>::TM rows);
// mc is the epilogue's output map, for epilogues that store by TMA.
template <class Epi, bool kF16, bool kWide = false>
static cudaError_t launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const GemmGeo& g,
                               const Epi& epi, int* dev_error, int sm_count, cudaStream_t st,
                               const CUtensorMap* mc = nullptr) {
    Problems<Epi> P;
    P.p[0].a = ma;
    P.p[0].b = mb;
    if (mc) P.p[0].c = *mc;
    P.p[0].g = g;
    P.p[0].epi = epi;
    P.p[1] = P.p[0];
    P.n0 = g.n_units;
    P.total = g.n_units;
    P.counter = nullptr;
    return launch_problems<Epi, kF16, 0u, kWide>(P, dev_error, sm_count, st);
}

// Two GEMMs in one launch, units claimed through `counter` (zeroed before),
// operand layouts kLayout, tile configuration kWide (the geometries' M tiles
// must be TileCfg<kWide>::TM rows).  The first problem should be the one with
// the longer units.
template <class Epi, bool kF16, uint32_t kLayout, bool kWide>
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
    return launch_problems<Epi, kF16, kLayout, kWide>(P, dev_error, sm_count, st);
}

static cudaError_t launch_to_fp16(const void* W, int64_t V, int64_t Vp, const void* hidden,
                                  const float* weights, int64_t T, int64_t Tp, int64_t d,
                                  __half* W16, __half* h16, int* dev_error, int sm_count,
                                  cudaStream_t st) {
    const int64_t nW8 = V * d / 8, nWp8 = Vp * d / 8, d8 = d / 8;
    const int64_t total = nWp8 + Tp * d8;
    int64_t grid = (total + 255) / 256;
    if (grid > (int64_t)sm_count * 8) grid = (int64_t)sm_count * 8;
    to_fp16_kernel<<<(unsigned)grid, 256, 0, st>>>(
        static_cast<const uint16_t*>(W), nW8, nWp8, W16, static_cast<const uint16_t*>(hidden),
        weights, T, Tp, d8, h16, dev_error);
    return cudaGetLastError();
}

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
    int64_t Vp;  // V padded to whole 64-row k-blocks (rows past V are zeros)
    size_t W16_off, h16_off, G_off, ctr_off, total;
    int64_t n_chunks;  // vocabulary chunks of VC columns
};
static BwdWorkspace bwd_layout(int64_t T, int64_t V, int64_t d) {
    BwdWorkspace w;
    // whole recompute tiles: a recompute tile writes every G row it covers
    constexpr int tm = TileCfg<GRAD_WIDE>::TM;
    w.Tp = (T + tm - 1) / tm * tm;
    w.Vp = (V + BK - 1) / BK * BK;
    w.W16_off = 0;                                                   // [Vp, d] fp16
    w.h16_off = align_up(w.W16_off + (size_t)w.Vp * d * 2, 1024);    // [Tp, d] fp16
    w.G_off = align_up(w.h16_off + (size_t)w.Tp * d * 2, 1024);      // [Tp, VC] fp16
    w.ctr_off = align_up(w.G_off + (size_t)w.Tp * VC * 2, 1024);     // int[n_chunks]
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
    constexpr int kFwdTM = lm::TileCfg<lm::FWD_WIDE>::TM;
    if (!lm::make_map(&map_h, false, hidden, T, d, d, kFwdTM) ||
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
    const lm::GemmGeo g = lm::geo(T, V, d, lm::STATS_TILES, 0, lm::M_GROUP, 0, kFwdTM);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (lm::launch_gemm<lm::StatsEpi, false, lm::FWD_WIDE>(map_h, map_w, g, epi, dev_error,
                                                           dev.sm_count, st) !=
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
    __half* W16 = reinterpret_cast<__half*>(ws + wl.W16_off);
    __half* h16 = reinterpret_cast<__half*>(ws + wl.h16_off);
    __half* G = reinterpret_cast<__half*>(ws + wl.G_off);
    const int64_t Tp = wl.Tp;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    // K-major maps (inner coordinate K): hidden and W for the recompute, G for
    // dhidden.  MN-major maps (inner coordinate M or N): G for dW (inner =
    // vocabulary), W16 for dhidden (inner = d) and h' for dW (inner = d).
    constexpr int kAccTM = lm::TileCfg<lm::ACC_WIDE>::TM;  // A rows per accumulation tile
    CUtensorMap map_h, map_w, map_Gst, map_G, map_Gmn, map_W16, map_h16;
    constexpr int kGradTM = lm::TileCfg<lm::GRAD_WIDE>::TM;
    if (!lm::make_map(&map_h, false, hidden, T, d, d, kGradTM) ||
        !lm::make_map(&map_w, false, W, V, d, d, lm::BN) ||
        // one epilogue warp's store: 32 rows x 64 columns of G
        !lm::make_map(&map_Gst, true, G, Tp, lm::VC, lm::VC, 32) ||
        !lm::make_map(&map_G, true, G, Tp, lm::VC, lm::VC, kAccTM) ||
        !lm::make_map_mn4d(&map_Gmn, G, Tp, lm::VC, lm::VC, kAccTM) ||
        !lm::make_map_mn4d(&map_W16, W16, wl.Vp, d, d, lm::BN) ||
        !lm::make_map_mn4d(&map_h16, h16, Tp, d, d, lm::BN))
        return PSTAT_ERR_CUDA;

    lm::GradEpi ge;
    ge.T = T;
    ge.V = V;
    ge.labels = labels;
    ge.ignore_index = ignore_index;
    ge.weights = weights;
    ge.rowstats = reinterpret_cast<const float2*>(rowstats);
    ge.dev_error = dev_error;

    const int64_t n_chunks = wl.n_chunks;
    int* ctr = reinterpret_cast<int*>(ws + wl.ctr_off);  // one unit counter per chunk
    if (cudaMemsetAsync(ctr, 0, (size_t)n_chunks * sizeof(int), st) != cudaSuccess)
        return PSTAT_ERR_CUDA;
    // 0. W16 = fp16(W), h' = fp16(w hidden)
    if (lm::launch_to_fp16(W, V, wl.Vp, hidden, weights, T, Tp, d, W16, h16, dev_error,
                           dev.sm_count, st) != cudaSuccess)
        return PSTAT_ERR_CUDA;

    for (int64_t c = 0; c < n_chunks; ++c) {
        const int64_t c0 = c * lm::VC;
        const int64_t vc = (V - c0) < lm::VC ? (V - c0) : lm::VC;
        // 1. recompute the chunk's logits -> G = fp16(-2^15 q)
        ge.c0 = c0;
        const lm::GemmGeo g1 = lm::geo(Tp, vc, d, 1, c0, lm::M_GROUP, 0, kGradTM);
        if (lm::launch_gemm<lm::GradEpi, false, lm::GRAD_WIDE>(map_h, map_w, g1, ge, dev_error,
                                                               dev.sm_count, st,
                                                               &map_Gst) != cudaSuccess)
            return PSTAT_ERR_CUDA;
        // 2. dhidden += (-w 2^-15) G W16_c  and  3. dW[c0 : c0 + vc] += -2^-15 G^T h',
        // in one launch: CTAs claim units of both GEMMs (the longer-K one
        // first) from this chunk's counter, so neither leaves a partial last
        // wave.
        lm::AccumEpi e2;
        e2.out = dhidden;
        e2.ld = d;
        e2.row0 = 0;
        e2.rows = T;
        e2.cols = d;
        e2.row_scale = weights;
        e2.scale = lm::GRAD_UNSCALE;
        const lm::GemmGeo g2 = lm::geo(T, d, vc, 1, 0, lm::ACC_M_GROUP, c0, kAccTM);
        lm::AccumEpi e3;
        e3.out = dW;
        e3.ld = d;
        e3.row0 = c0;
        e3.rows = vc;
        e3.cols = d;
        e3.row_scale = nullptr;
        e3.scale = lm::GRAD_UNSCALE;
        const lm::GemmGeo g3 = lm::geo(vc, d, Tp, 1, 0, lm::ACC_M_GROUP, 0, kAccTM);
        // dW: A and B MN-major; dhidden: A K-major, B MN-major
        constexpr uint32_t kDwFirst = lm::layout_bits(1, 1, 0, 1);
        constexpr uint32_t kDhFirst = lm::layout_bits(0, 1, 1, 1);
        const cudaError_t e =
            g3.k_blocks >= g2.k_blocks
                ? lm::launch_gemm_pair<lm::AccumEpi, true, kDwFirst, lm::ACC_WIDE>(
                      map_Gmn, map_h16, g3, e3, map_G, map_W16, g2, e2, ctr + c, dev_error,
                      dev.sm_count, st)
                : lm::launch_gemm_pair<lm::AccumEpi, true, kDhFirst, lm::ACC_WIDE>(
                      map_G, map_W16, g2, e2, map_Gmn, map_h16, g3, e3, ctr + c, dev_error,
                      dev.sm_count, st);
        if (e != cudaSuccess) return PSTAT_ERR_CUDA;
    }
    return PSTAT_OK;
}

}  // extern "C"
