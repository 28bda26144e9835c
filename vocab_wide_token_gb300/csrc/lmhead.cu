// lmhead.cu -- fused lm_head statistics on the 5th-generation tensor cores.
//
// Logits z = hidden W^T are produced tile by tile (128 tokens x 256 vocab
// rows, K = d in steps of 64) by tcgen05.mma into tensor memory and folded
// straight into the per-(token, 4096-column chunk) statistics (m, s, u) that
// the unfused path also produces; the logits never reach global memory.  The
// fixed-order combine kernel then turns the chunk statistics into logprob,
// entropy and (M, ln S).  The chunked lm_head follows TRL PR #6949
// ("ZeroSyncGRPOTrainer": the vocabulary projection is multiplied chunk by
// chunk; GEMMs in bf16 with fp32 accumulation).
//
// CTA roles (192 threads, one CTA per SM):
//   warp 0     TMA producer: 2-D tiled loads of hidden and W k-blocks into a
//              4-stage shared-memory ring (128-byte swizzle)
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators)
//              and issues the MMAs from one thread
//   warps 2-5  epilogue: one thread per token row reads its accumulator row
//              from TMEM and folds it into the chunk statistics
// All waits are bounded; a timeout sets PSTAT_DEV_TIMEOUT and the CTA winds
// down, draining its copies and MMAs before freeing tensor memory.
#include <cuda.h>
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

constexpr int BM = 128;            // tokens per tile (MMA M, TMEM lanes)
constexpr int BN = 256;            // vocabulary rows per tile (MMA N)
constexpr int BK = 64;             // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int UK = 16;             // K per tcgen05.mma of kind::f16
constexpr int STAGES = 4;
constexpr int TILES_PER_CHUNK = PSTAT_CHUNK_BF16 / BN;  // 16
constexpr int M_GROUP = 32;        // m-tiles sharing the L2-resident slice of hidden
constexpr int THREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;   // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 2 * BN;      // double-buffered accumulator
constexpr uint64_t WAIT_NS = 2000000000ull;

struct Smem {
    // Offsets inside the 1024-byte aligned dynamic shared memory block.
    static constexpr uint32_t a = 0;
    static constexpr uint32_t b = a + STAGES * A_BYTES;
    static constexpr uint32_t bars = b + STAGES * B_BYTES;
    // full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
    static constexpr uint32_t n_bars = 2 * STAGES + 4 + 1;
    static constexpr uint32_t tmem_slot = bars + n_bars * 8;
    static constexpr uint32_t total = tmem_slot + 16;
};
constexpr size_t SMEM_BYTES = Smem::total + 1024;  // + alignment slack

struct Geometry {
    int64_t T, V;
    int d;
    int m_tiles, n_tiles, n_chunks, k_blocks;
    int64_t n_units;
};

__host__ __device__ inline void unit_coords(const Geometry& g, int64_t u, int& m, int& c) {
    const int64_t per_group = (int64_t)M_GROUP * g.n_chunks;
    const int grp = (int)(u / per_group);
    const int64_t rem = u - (int64_t)grp * per_group;
    int mg = g.m_tiles - grp * M_GROUP;
    if (mg > M_GROUP) mg = M_GROUP;
    c = (int)(rem / mg);
    m = grp * M_GROUP + (int)(rem % mg);
}

__device__ __forceinline__ int tiles_in_chunk(const Geometry& g, int c) {
    const int nt = g.n_tiles - c * TILES_PER_CHUNK;
    return nt < TILES_PER_CHUNK ? nt : TILES_PER_CHUNK;
}

// Folds tile statistics (mj, sj, uj) into the running chunk statistics.
__device__ __forceinline__ void fold(float& mc, float& sc, float& uc, float mj, float sj, float uj) {
    if (mj == -INFINITY) return;
    if (mc == -INFINITY) {
        mc = mj;
        sc = sj;
        uc = uj;
        return;
    }
    if (mj > mc) {
        const float dm = mc - mj;
        const float r = expf(dm);
        uc = r * fmaf(dm, sc, uc);
        sc = r * sc;
        mc = mj;
        sc += sj;
        uc += uj;
    } else {
        const float dm = mj - mc;
        const float r = expf(dm);
        sc = fmaf(r, sj, sc);
        uc = fmaf(r, fmaf(dm, sj, uj), uc);
    }
}

__global__ void __launch_bounds__(THREADS, 1)
    lmhead_stats_kernel(const __grid_constant__ CUtensorMap map_h,
                        const __grid_constant__ CUtensorMap map_w, const Geometry g,
                        const int64_t* __restrict__ labels, int64_t ignore_index,
                        float4* __restrict__ chunk_stats, float* __restrict__ target,
                        int* __restrict__ dev_error) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Smem::bars);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Smem::tmem_slot);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

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
        fence_mbar_init();
        prefetch_tensormap(&map_h);
        prefetch_tensormap(&map_w);
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

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            const uint64_t pol_h = policy_evict_last();
            const uint64_t pol_w = policy_evict_first();
            uint32_t it = 0;
            for (int64_t u = blockIdx.x; u < g.n_units && !failed; u += gridDim.x) {
                int m, c;
                unit_coords(g, u, m, c);
                const int nt = tiles_in_chunk(g, c);
                for (int j = 0; j < nt && !failed; ++j) {
                    const int n = c * TILES_PER_CHUNK + j;
                    for (int kb = 0; kb < g.k_blocks; ++kb, ++it) {
                        const int s = it % STAGES;
                        const uint32_t ph = (it / STAGES) & 1u;
                        if (!mbar_wait_bounded(&empty[s], ph ^ 1u, WAIT_NS)) {
                            failed = true;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                        tma_load_2d(smem + Smem::a + s * A_BYTES, &map_h, kb * BK, m * BM,
                                    &full[s], pol_h);
                        tma_load_2d(smem + Smem::b + s * B_BYTES, &map_w, kb * BK, n * BN,
                                    &full[s], pol_w);
                    }
                }
            }
            // Every copy this thread issued must have landed before the CTA can
            // end (on the normal path they all have; after a timeout some may not).
            for (uint32_t k = 0; k < (uint32_t)STAGES && k < it; ++k) {
                const uint32_t i = it - 1 - k;
                if (!mbar_wait_bounded(&full[i % STAGES], (i / STAGES) & 1u, WAIT_NS)) failed = true;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
            uint32_t it = 0, tc = 0;
            for (int64_t u = blockIdx.x; u < g.n_units && !failed; u += gridDim.x) {
                int m, c;
                unit_coords(g, u, m, c);
                const int nt = tiles_in_chunk(g, c);
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
        // ---------------- epilogue: statistics ----------------
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int row = q * 32 + lane;
        const uint64_t l2e = f2_pack(kLog2e, kLog2e);
        uint32_t tc = 0;
        for (int64_t u = blockIdx.x; u < g.n_units && !failed; u += gridDim.x) {
            int m, c;
            unit_coords(g, u, m, c);
            const int nt = tiles_in_chunk(g, c);
            const int64_t t = (int64_t)m * BM + row;
            const bool valid_t = t < g.T;
            const int64_t y = (valid_t && labels) ? labels[t] : ignore_index;
            float mc = -INFINITY, sc = 0.f, uc = 0.f;
            for (int j = 0; j < nt; ++j, ++tc) {
                const int64_t col0 = (int64_t)(c * TILES_PER_CHUNK + j) * BN;
                const int64_t left = g.V - col0;
                const int ncols = left < BN ? (int)left : BN;
                const uint32_t b = tc & 1u;
                const uint32_t tph = (tc >> 1) & 1u;
                bool ok = mbar_wait_bounded(&tfull[b], tph, WAIT_NS);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) {
                    failed = true;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + b * BN;
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
                uint64_t s2 = 0, u2 = 0;
                float zy = 0.f;
                bool have_y = false;
                const int64_t yl = y - col0;
                for (int p = 0; p < BN / 32; ++p) {
                    if (p * 32 >= ncols) break;
                    float v[32];
                    tmem_ld32(taddr + p * 32, v);
                    tmem_ld_wait();
                    if (yl >= p * 32 && yl < p * 32 + 32 && yl < ncols) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (yl == p * 32 + i) zy = v[i];
                        have_y = true;
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
                // accumulator b may be overwritten from here on
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[b]);
                float sa, sb, ua, ub;
                f2_unpack(s2, sa, sb);
                f2_unpack(u2, ua, ub);
                fold(mc, sc, uc, mx, sa + sb, ua + ub);
                if (have_y && valid_t) target[t] = zy;
            }
            if (failed) break;
            if (valid_t) chunk_stats[t * g.n_chunks + c] = make_float4(mc, sc, uc, 0.f);
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
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Row-major bf16 matrix [rows, cols] -> tensor map with box [box_rows, 64].
static bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t cols,
                     int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static Geometry geometry(int64_t T, int64_t V, int64_t d) {
    Geometry g;
    g.T = T;
    g.V = V;
    g.d = (int)d;
    g.m_tiles = (int)((T + BM - 1) / BM);
    g.n_tiles = (int)((V + BN - 1) / BN);
    g.n_chunks = (int)((V + PSTAT_CHUNK_BF16 - 1) / PSTAT_CHUNK_BF16);
    g.k_blocks = (int)(d / BK);
    g.n_units = (int64_t)g.m_tiles * g.n_chunks;
    return g;
}

struct LmWorkspace {
    size_t stats_off, target_off, total;
};
static LmWorkspace lm_layout(int64_t T, int64_t V) {
    const int64_t nc = (V + PSTAT_CHUNK_BF16 - 1) / PSTAT_CHUNK_BF16;
    LmWorkspace w;
    w.stats_off = 0;
    w.target_off = align_up((size_t)T * nc * kChunkRecordBytes, 256);
    w.total = align_up(w.target_off + (size_t)T * sizeof(float), 256);
    return w;
}

static int check_lm_args(const void* hidden, const void* W, int64_t T, int64_t V, int64_t d) {
    if (T < 0 || V < 1 || d < BK || d % BK != 0 || d > (1 << 20)) return PSTAT_ERR_SHAPE;
    if (T > (int64_t)INT32_MAX || V > (int64_t)INT32_MAX) return PSTAT_ERR_SHAPE;
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
    *bytes = lm::lm_layout(T, V).total;
    return PSTAT_OK;
}

int pstat_lmhead_fused(const void* hidden, const void* W, int64_t T, int64_t V, int64_t d,
                       const int64_t* labels, int64_t ignore_index, float* out_logprob,
                       float* out_entropy, float* out_rowstats, void* workspace,
                       size_t ws_bytes, int* dev_error, pstat_stream_t stream) {
    int rc = lm::check_lm_args(hidden, W, T, V, d);
    if (rc != PSTAT_OK || T == 0) return rc;
    const lm::LmWorkspace wl = lm::lm_layout(T, V);
    if (!workspace || ws_bytes < wl.total) return PSTAT_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 15u) return PSTAT_ERR_ALIGN;
    if ((labels && (reinterpret_cast<uintptr_t>(labels) & 7u)) ||
        (out_rowstats && (reinterpret_cast<uintptr_t>(out_rowstats) & 7u)))
        return PSTAT_ERR_ALIGN;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    ShardPlan plan;
    rc = make_plan(V, PSTAT_CHUNK_BF16, nullptr, 1, &plan);
    if (rc != PSTAT_OK) return rc;

    CUtensorMap map_h, map_w;
    if (!lm::make_map(&map_h, hidden, T, d, lm::BM) || !lm::make_map(&map_w, W, V, d, lm::BN))
        return PSTAT_ERR_CUDA;
    const lm::Geometry g = lm::geometry(T, V, d);
    char* ws = static_cast<char*>(workspace);
    float4* cs = reinterpret_cast<float4*>(ws + wl.stats_off);
    float* target = reinterpret_cast<float*>(ws + wl.target_off);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    static std::atomic<bool> configured[64];
    int devi = 0;
    cudaGetDevice(&devi);
    if (devi >= 64 || !configured[devi].load()) {
        if (cudaFuncSetAttribute(lm::lmhead_stats_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)lm::SMEM_BYTES) != cudaSuccess)
            return PSTAT_ERR_CUDA;
        if (devi < 64) configured[devi].store(true);
    }
    int64_t grid = g.n_units < dev.sm_count ? g.n_units : dev.sm_count;
    lm::lmhead_stats_kernel<<<(unsigned)grid, lm::THREADS, lm::SMEM_BYTES, st>>>(
        map_h, map_w, g, labels, ignore_index, cs, target, dev_error);
    if (cudaGetLastError() != cudaSuccess) return PSTAT_ERR_CUDA;
    if (launch_combine(cs, plan, nullptr, PSTAT_BF16, T, V, V, labels, ignore_index, target,
                       out_logprob, out_entropy, out_rowstats, dev_error, st) != cudaSuccess)
        return PSTAT_ERR_CUDA;
    return PSTAT_OK;
}

int pstat_lmhead_backward(const void* hidden, const void* W, int64_t T, int64_t V, int64_t d,
                          const int64_t* labels, int64_t ignore_index, const float* weights,
                          const float* rowstats, float* dhidden, float* dW, void* workspace,
                          size_t ws_bytes, int* dev_error, pstat_stream_t stream) {
    (void)hidden; (void)W; (void)T; (void)V; (void)d; (void)labels; (void)ignore_index;
    (void)weights; (void)rowstats; (void)dhidden; (void)dW; (void)workspace; (void)ws_bytes;
    (void)dev_error; (void)stream;
    return PSTAT_ERR_UNSUPPORTED;
}

}  // extern "C"
