// fused.cu -- pstat_forward_backward: logprob, entropy, (M, ln S) and the
// weighted backward dlogits = w (onehot(y) - softmax(z)) in one kernel.
//
// Calling pstat_forward then pstat_backward streams the logits from HBM
// twice (6V bytes per bf16 token with the dlogits write).  Here each CTA owns
// whole rows and passes over every row twice back to back:
//   pass 1  streams the row's chunks from HBM (bulk copies with an L2
//           evict-last hint) and forms each chunk's (m, s, u) record, exactly
//           as the chunk-statistics kernel does, into shared memory;
//           the warp that finishes the row's last chunk folds the records in
//           the fixed order of the combine kernel and publishes (M, ln S);
//   pass 2  takes the same chunks again -- the warp's last one still in its
//           registers, the one before still in its bulk-copy slot, the rest
//           re-read from L2 -- and writes dlogits with the element-wise
//           arithmetic of the backward kernel.
// HBM sees 4V bytes per token (read once, write once).  Rows are dealt to
// CTAs round robin; each warp keeps its 2-slot ring of bulk copies full
// across both passes and across rows.  (Running pass 1 of the next row before
// pass 2 of the current one hides the fold, but doubles the rows each SM
// keeps in L2, and pass 2 then misses L2: measured slower.)  Every record, fold
// and gradient element is computed by the same code as in the two-call path,
// so the results are bit-identical to pstat_forward + pstat_backward.
//
// The same kernel without pass 2 is pstat_forward's one-kernel path (for
// plans of at most 256 chunks per row): pass 1 with an evict-first hint, and
// the rows folded by the warps with one chunk less, or, when every warp holds
// as many chunks, by a fourteenth warp of its own, so that no warp's next row
// waits for a fold.  fp32 rows too wide for L2 on every SM run the single pass
// on three quarters of the SMs.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "chunk_math.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace pstat {
namespace {

constexpr int kFbMaxChunks = 256;  // chunk records per row held in shared memory
// Warps per CTA.  13 rather than the 12 of the chunk-statistics kernel: a
// 38-chunk row then splits 3 / 3 / ... / 2 over the warps instead of
// 4 / 4 / 3 / ... / 3, and every row waits for its slowest warp.
constexpr int kFbWarps = 13;
constexpr int kFbStages = 2;  // bulk-copy slots per warp

struct RowInfo {
    GradRow gr;  // gradient constants from (M, ln S, w) (mode 2)
    int mode;    // 0: all-zero row, 1: NaN row, 2: compute
    float zy;    // the label's logit (mode 2)
    long long y;
};

constexpr size_t kRingBytes = (size_t)kFbWarps * kFbStages * kSlotBytes;
constexpr size_t kBarBytes = (size_t)kFbWarps * kFbStages * sizeof(uint64_t);
constexpr size_t kRecOff = (kRingBytes + kBarBytes + 15) / 16 * 16;  // float4 records
constexpr size_t kInfoOff = kRecOff + 2 * kFbMaxChunks * sizeof(float4);
constexpr size_t kReadyOff = kInfoOff + 2 * sizeof(RowInfo);
constexpr size_t kRecsOff = kReadyOff + 2 * sizeof(uint64_t);  // forward only
constexpr size_t kCountOff = kRecsOff + 2 * sizeof(uint64_t);
// Labels, weights and label logits z_y of the CTA's first kFbRowCache rows,
// loaded once at the start so that the fold finds them in shared memory (a
// global load of z_y in the fold would put its latency on every row's
// critical path).
constexpr int kFbRowCache = 384;
constexpr size_t kLabOff = (kCountOff + 2 * sizeof(int) + 7) / 8 * 8;
constexpr size_t kWtOff = kLabOff + kFbRowCache * sizeof(int64_t);
constexpr size_t kZyOff = kWtOff + kFbRowCache * sizeof(float);
constexpr size_t kFusedSmem = kZyOff + kFbRowCache * sizeof(float);
static_assert(kRingBytes % 16 == 0 && kRecOff % 16 == 0, "slots and records: 16-byte aligned");
static_assert(kInfoOff % 8 == 0 && kReadyOff % 8 == 0, "RowInfo and mbarriers: 8-byte aligned");

template <typename E>
struct OutVec;
template <>
struct OutVec<uint16_t> {  // bf16 output, round to nearest even
    template <int N>
    __device__ static void store(uint16_t* p, const float (&g)[N]) {
        if constexpr (N == 8) {
            uint4 q;
            q.x = bf2_pack_rn(g[0], g[1]);
            q.y = bf2_pack_rn(g[2], g[3]);
            q.z = bf2_pack_rn(g[4], g[5]);
            q.w = bf2_pack_rn(g[6], g[7]);
            __stcs(reinterpret_cast<uint4*>(p), q);
        } else {
            uint2 q;
            q.x = bf2_pack_rn(g[0], g[1]);
            q.y = bf2_pack_rn(g[2], g[3]);
            __stcs(reinterpret_cast<uint2*>(p), q);
        }
    }
    __device__ static uint16_t one(float g) { return (uint16_t)(bf2_pack_rn(g, 0.f) & 0xFFFFu); }
};
template <>
struct OutVec<float> {
    template <int N>
    __device__ static void store(float* p, const float (&g)[N]) {
#pragma unroll
        for (int i = 0; i < N; i += 4)
            __stcs(reinterpret_cast<float4*>(p + i), make_float4(g[i], g[i + 1], g[i + 2], g[i + 3]));
    }
    __device__ static float one(float g) { return g; }
};

// The backward kernel's element arithmetic for N = 4 or 8 elements (N = 4:
// the fp32 vector is evaluated as the first half of an 8-element one).
template <int N>
__device__ __forceinline__ void exp_vec(const float (&x)[N], const GradRow& r, float (&e)[N]) {
    if constexpr (N == 8) {
        exp8(x, r.m2, e);
    } else {
        float x8[8] = {x[0], x[1], x[2], x[3], x[0], x[1], x[2], x[3]};
        float e8[8];
        exp8(x8, r.m2, e8);
#pragma unroll
        for (int i = 0; i < N; ++i) e[i] = e8[i];
    }
}
template <int N>
__device__ __forceinline__ void grad_vec(const float (&x)[N], const RowInfo& ri, int64_t col0,
                                         int64_t y, float (&g)[N]) {
    float e[N];
    exp_vec<N>(x, ri.gr, e);
    const uint64_t k = f2_pack(ri.gr.nwK, ri.gr.nwK);
#pragma unroll
    for (int i = 0; i < N; i += 2) f2_unpack(f2_mul(f2_pack(e[i], e[i + 1]), k), g[i], g[i + 1]);
    const int64_t r = y - col0;
    if (r >= 0 && r < N) {
#pragma unroll
        for (int i = 0; i < N; ++i)
            if (i == r) g[i] = grad_label(e[i], ri.gr);  // w (1 - p_y)
    }
}

// Same without the label column (the caller knows it is not in the vector).
template <int N>
__device__ __forceinline__ void grad_vec_nolabel(const float (&x)[N], const RowInfo& ri,
                                                 float (&g)[N]) {
    float e[N];
    exp_vec<N>(x, ri.gr, e);
    const uint64_t k = f2_pack(ri.gr.nwK, ri.gr.nwK);
#pragma unroll
    for (int i = 0; i < N; i += 2) f2_unpack(f2_mul(f2_pack(e[i], e[i + 1]), k), g[i], g[i + 1]);
}

template <typename Ein>
__device__ __forceinline__ void unpack_vec(const uint4& v, float (&x)[Elem<Ein>::kVec]);
template <>
__device__ __forceinline__ void unpack_vec<uint16_t>(const uint4& v, float (&x)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = bf2_lo(w[i]);
        x[2 * i + 1] = bf2_hi(w[i]);
    }
}
template <>
__device__ __forceinline__ void unpack_vec<float>(const uint4& v, float (&x)[4]) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
}

// kBwd = false: pass 1 only (the forward: logprob, entropy, (M, ln S)).
// kShard (forward only): the per-shard statistics instead of the row outputs.
// kShards (with the backward): a plan of several shards, whose rows hold
// several chunks shorter than a full one.
// kOwnFolder (forward only): one more warp, which owns no chunk and folds the
// rows, for plans in which every chunk-owning warp holds as many chunks.
template <typename Ein, typename Eout, bool kBwd, bool kShard = false, bool kShards = false,
          bool kOwnFolder = false>
__global__ void __launch_bounds__((kFbWarps + (kOwnFolder ? 1 : 0)) * 32, 1)
    fwdbwd_kernel(const Ein* __restrict__ logits, int64_t T, int64_t V, int64_t ld,
                  const __grid_constant__ ShardPlan plan, const int64_t* __restrict__ labels,
                  int64_t ignore_index, const float* __restrict__ weights,
                  float* __restrict__ logprob, float* __restrict__ entropy,
                  float* __restrict__ rowstats, Eout* __restrict__ out, int64_t ld_out,
                  float4* __restrict__ shard_out, int64_t label_offset,
                  int* __restrict__ dev_error) {
    // shard_out (forward only): instead of the row outputs, write the row's
    // statistics (M, S, U, z_y) for this vocabulary shard, whose first column
    // is label_offset in the labels' numbering; z_y is 0 when the label lies
    // outside the shard.
    constexpr int kVec = Elem<Ein>::kVec;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* slots = smem + (size_t)warp * kFbStages * kSlotBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRingBytes) + warp * kFbStages;
    float4* records = reinterpret_cast<float4*>(smem + kRecOff);
    RowInfo* info = reinterpret_cast<RowInfo*>(smem + kInfoOff);
    uint64_t* ready = reinterpret_cast<uint64_t*>(smem + kReadyOff);
    uint64_t* recs = reinterpret_cast<uint64_t*>(smem + kRecsOff);
    int* counter = reinterpret_cast<int*>(smem + kCountOff);
    int64_t* lab_s = reinterpret_cast<int64_t*>(smem + kLabOff);
    float* wt_s = reinterpret_cast<float*>(smem + kWtOff);
    float* zy_s = reinterpret_cast<float*>(smem + kZyOff);

    const int nc = plan.n_chunks;
    const int active = nc < kFbWarps ? nc : kFbWarps;  // warps that own chunks of any one row
    // Forward only: the warps with the fewest chunks per row, [active - n_fold,
    // active), take turns folding the rows (with kOwnFolder, warp 13 does).
    const int n_fold = nc >= kFbWarps && nc % kFbWarps != 0 ? kFbWarps - nc % kFbWarps : active;
    if (lane == 0 && (!kOwnFolder || warp < kFbWarps)) {
        for (int s = 0; s < kFbStages; ++s) mbar_init(&bars[s], 1);
    }
    if (threadIdx.x == 0) {
        mbar_init(&ready[0], 1);
        mbar_init(&ready[1], 1);
        // forward only: the records of the row's other chunk-owning warps
        // (all of them with a folding warp of its own) are in
        const int others = kOwnFolder ? active : active - 1;
        mbar_init(&recs[0], others > 0 ? others : 1);
        mbar_init(&recs[1], others > 0 ? others : 1);
        counter[0] = 0;
        counter[1] = 0;
    }
    const int64_t nrows = (T > (int64_t)blockIdx.x) ? (T - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
    for (int64_t r = threadIdx.x; r < nrows && r < kFbRowCache; r += blockDim.x) {
        const int64_t t = blockIdx.x + r * gridDim.x;
        const int64_t y = labels ? labels[t] : ignore_index;
        lab_s[r] = y;
        wt_s[r] = weights ? weights[t] : 1.f;
        const int64_t yl = kShard ? y - label_offset : y;  // the label's column here
        zy_s[r] = (y != ignore_index && yl >= 0 && yl < V) ? Elem<Ein>::to_float(logits[t * ld + yl])
                                                           : 0.f;
    }
    fence_mbar_init();
    __syncthreads();
    // Both passes of row k: warp w owns chunks g = w, w + 13, ... .  Pass 2
    // takes them starting with the last one, which is still in the warp's
    // registers from pass 1, then the one before it, which is still in its
    // bulk-copy slot (the refill that would have overwritten it is skipped:
    // with two slots, pass 2's second copy position falls on exactly that
    // slot), then the others in order, re-read from L2.
    // With at least 13 chunks every warp owns chunks of every row, so it
    // arrives for every row's fold and reads every row's statistics before the
    // double-buffered records and row data are reused two rows later.  With
    // fewer chunks warps without a chunk leave (warp 13 of kOwnFolder owns
    // none and stays: it folds every row as soon as its records are in).
    if (nc < kFbWarps && warp >= nc && (!kOwnFolder || warp < kFbWarps)) return;

    const uint64_t pol_keep = policy_evict_last();
    const uint64_t pol_once = policy_evict_first();

    // A warp's work is the sequence of segments pass 1 of row k, pass 2 of
    // row k, for the CTA's rows k = 0, 1, ... in order (pass 1 only without
    // the backward).
    struct Cursor {
        int64_t k;
        int pass, i, cnt, g0;
    };
    auto load_segment = [&](Cursor& c) {
        if (c.k >= nrows) {
            c.cnt = 0;
            return;
        }
        c.g0 = warp;
        c.cnt = c.g0 < nc ? (nc - c.g0 + kFbWarps - 1) / kFbWarps : 0;
    };
    auto settle = [&](Cursor& c) {  // first position at or after c that holds a chunk
        while (c.k < nrows) {
            load_segment(c);
            if (c.i < c.cnt) return;
            c.i = 0;
            if (c.pass == 0 && kBwd) {
                c.pass = 1;
            } else {
                c.pass = 0;
                ++c.k;
            }
        }
    };
    auto advance = [&](Cursor& c) {
        ++c.i;
        settle(c);
    };
    auto done = [&](const Cursor& c) { return c.k >= nrows; };
    // Pass 2's first position is the chunk pass 1 left in registers (no slot);
    // its second is the chunk pass 1 left in its slot (no copy).
    static_assert(kFbStages == 2, "the slot-held chunk relies on a 2-slot ring");
    auto held = [&](const Cursor& c) { return kBwd && c.pass == 1 && c.i == 0; };
    auto in_slot = [&](const Cursor& c) { return kBwd && c.pass == 1 && c.i == 1; };
    auto advance_issue = [&](Cursor& c) {  // next position that uses a slot
        advance(c);
        if (!done(c) && held(c)) advance(c);
    };

    struct Task {
        int64_t r, t;  // the CTA's row index, token row
        int g;
        bool bulk;     // served by a bulk copy into its slot
        const Ein* src;
        int64_t start;
        int len;
    };
    auto task_of = [&](const Cursor& c) {
        Task tk;
        tk.r = c.k;
        const int j = c.pass == 0 ? c.i : c.i == 0 ? c.cnt - 1 : c.i == 1 ? c.cnt - 2 : c.i - 2;
        tk.g = c.g0 + kFbWarps * j;
        tk.t = blockIdx.x + tk.r * gridDim.x;
        chunk_span(plan, tk.g, tk.start, tk.len);
        tk.src = logits + tk.t * ld + tk.start;
        tk.bulk = ((reinterpret_cast<uintptr_t>(tk.src) & 15u) == 0) &&
                  ((((size_t)tk.len * sizeof(Ein)) & 15u) == 0);
        return tk;
    };
    auto issue = [&](const Cursor& c, int64_t pos) {
        const Task tk = task_of(c);
        if (tk.bulk && lane == 0) {
            const int slot = (int)(pos % kFbStages);
            const uint32_t bytes = (uint32_t)tk.len * (uint32_t)sizeof(Ein);
            // Pass 1 of the single pass: pass 2 reads the chunk again from L2,
            // so keep it there.  A warp's last two chunks of a row are not read
            // again (pass 2 takes them from registers and from their slot); for
            // fp32 rows they are loaded evict-first, which leaves more of L2 to
            // the others (1.635 -> 1.616 ms at V = 151,936; for bf16 the same
            // measured 0.7% slower).
            const bool keep =
                kBwd && c.pass == 0 && (sizeof(Ein) == 2 || c.i < c.cnt - 2);
            mbar_arrive_expect_tx(&bars[slot], bytes);
            bulk_g2s_hint(slots + (size_t)slot * kSlotBytes, tk.src, bytes, &bars[slot],
                          keep ? pol_keep : pol_once);
        }
    };

    if constexpr (kOwnFolder) {
        // The fold of the CTA's r-th row, token row t, whose chunk records are
        // in records[b]: the row's statistics in the combine kernel's order,
        // then what pass 2 needs, published on ready[b], then the row outputs.
        // Called by the forward's folding warp; the chunk loop below writes
        // the same steps out in place.
        auto fold_row = [&](int64_t r, int64_t t, int b) {
            __threadfence_block();
            // Label, weight and z_y first (for rows past the cache
            // the z_y load then runs under the fold's arithmetic).
            const bool cached = r < kFbRowCache;
            const int64_t y = cached ? lab_s[r] : (labels ? labels[t] : ignore_index);
            const float w = cached ? wt_s[r] : (weights ? weights[t] : 1.f);
            const int64_t yl = kShard ? y - label_offset : y;  // the label's column here
            const bool y_in = y != ignore_index && yl >= 0 && yl < V;
            float zy = 0.f;
            if (lane == 0 && y_in)
                zy = cached ? zy_s[r] : Elem<Ein>::to_float(logits[t * ld + yl]);
            const float3 st = fold_row_warp(records + b * kFbMaxChunks, plan, lane);
            if (kShard && lane == 0) {
                shard_out[t] = make_float4(st.x, st.y, st.z, zy);
                mbar_arrive(&ready[b]);
            } else if (lane == 0) {
                counter[b] = 0;
                const float M = st.x, S = st.y, U = st.z;
                // First what pass 2 waits for -- ln S, the row's mode and
                // its gradient constants -- then publish; the entropy
                // (a division) and the global stores come after.
                const bool empty = !(M > -INFINITY);
                const bool bad = !empty && y != ignore_index && (y < 0 || y >= V);
                const float lnS = empty ? NAN : logf(S);
                RowInfo nr;
                nr.mode = (y == ignore_index || w == 0.f) ? 0 : (empty || bad) ? 1 : 2;
                nr.gr = nr.mode == 2 ? grad_row(M, lnS, w) : GradRow{0.f, 0.f, 0.f, 0.f};
                nr.y = y;
                nr.zy = zy;
                info[b] = nr;
                mbar_arrive(&ready[b]);  // release: records, info visible to waiters
                float H, lp;
                if (empty) {
                    H = NAN;
                    lp = NAN;
                } else {
                    H = lnS - U / S;
                    if (y == ignore_index) {
                        lp = 0.f;
                    } else if (bad) {
                        lp = NAN;
                        H = NAN;
                    } else {
                        lp = (zy - M) - lnS;
                    }
                }
                if (logprob) logprob[t] = lp;
                if (entropy) entropy[t] = H;
                if (rowstats) reinterpret_cast<float2*>(rowstats)[t] = make_float2(M, lnS);
                const int err = (empty ? PSTAT_DEV_EMPTY_ROW : 0) | (bad ? PSTAT_DEV_BAD_LABEL : 0);
                if (err && dev_error) atomicOr(dev_error, err);
            }
        };

        if (warp == kFbWarps) {
            // The folding warp.  With every chunk warp holding as many chunks
            // of a row, a chunk warp that folded would wait for the others'
            // records (warps drift up to two rows apart) and start its next
            // row late: 3-shard forward 0.465 against 0.411 ms.
            for (int64_t r = 0; r < nrows; ++r) {
                const int b = (int)(r & 1);
                bool ok = mbar_wait_bounded(&recs[b], (uint32_t)((r >> 1) & 1), kWaitLimitNs);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) {
                    if (lane == 0 && dev_error) atomicOr(dev_error, PSTAT_DEV_TIMEOUT);
                    return;
                }
                fold_row(r, blockIdx.x + r * gridDim.x, b);
                __syncwarp();
            }
            return;
        }
    }

    Cursor ci = {0, 0, 0, 0, 0};  // next position to issue
    settle(ci);
    int64_t pi = 0;
    for (int s = 0; s < kFbStages && !done(ci); ++s, ++pi) {
        if (!in_slot(ci)) issue(ci, pi);
        advance_issue(ci);
    }

    Cursor cc = {0, 0, 0, 0, 0};  // position being consumed
    settle(cc);
    int64_t pc = 0;
    uint32_t phase = 0;  // parity bit per ring slot
    bool failed = false;
    RowInfo ri = {{0.f, 0.f, 0.f, 0.f}, 0, 0.f, 0};
    uint4 q[kVecPerLane];  // the chunk being processed; kept across positions for pass 2
    bool row_inf = false;  // this warp's first chunk of the current row held a -inf
    while (!done(cc)) {
        const Task tk = task_of(cc);
        const bool hold = held(cc);     // data already in q
        const bool kept = in_slot(cc);  // data already in this slot
        const int b = (int)(tk.r & 1);
        const int slot = (int)(pc % kFbStages);
        Ein* buf = reinterpret_cast<Ein*>(slots + (size_t)slot * kSlotBytes);
        const int len = tk.len;
        const int64_t start = tk.start;

        if (!kBwd && cc.i == 0 && tk.r >= 2) {
            // Forward only: the records, counter and row slot of parity b are
            // reused once row r - 2 is folded (nothing else holds warps within
            // a row of each other).
            bool ok = mbar_wait_bounded(&ready[b], (uint32_t)(((tk.r - 2) >> 1) & 1), kWaitLimitNs);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) {
                failed = true;
                break;
            }
        }
        if (kBwd && cc.pass == 1 && cc.i == 0) {
            // (M, ln S) of this row, published by the warp that folded it.
            bool ok = mbar_wait_bounded(&ready[b], (uint32_t)((tk.r >> 1) & 1), kWaitLimitNs);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) {
                failed = true;
                break;
            }
            ri = info[b];
        }
        const bool need_data = cc.pass == 0 || ri.mode == 2;
        if (!hold) {
            if (kept) {
                // left in the slot by pass 1; no copy was issued for it
            } else if (tk.bulk) {
                bool ok = mbar_wait_bounded(&bars[slot], (phase >> slot) & 1u, kWaitLimitNs);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) {
                    failed = true;
                    break;
                }
                phase ^= 1u << slot;
            } else if (need_data) {
                // Unaligned chunk: element loads, padded with -inf to a whole vector.
                const int padded = (len + kVec - 1) / kVec * kVec;
                for (int k = lane; k < padded; k += 32)
                    buf[k] = (k < len) ? tk.src[k] : Elem<Ein>::neg_inf();
                __syncwarp();
            }
            if (need_data) load_chunk_regs<Ein>(buf, len, lane, q);
            __syncwarp();
            fence_proxy_async_smem();  // our reads of the slot precede the next bulk write into it
            if (!done(ci)) {
                if (!in_slot(ci)) issue(ci, pi);
                advance_issue(ci);
                ++pi;
            }
        }
        const int nvec = (len + kVec - 1) / kVec;

        if (cc.pass == 0) {
            // A short chunk goes straight to the clamped pass, and so does a
            // warp's later chunk of a row whose first chunk held a -inf (masked
            // rows hold them throughout), except in the single pass over a
            // one-shard plan, where that form measured 0.6% slower (same bits).
            constexpr bool kPredict = !kBwd || kShards;
            bool had_inf = false;
            const float4 rec = reduce_regs(q, (Ein*)nullptr,
                                           kPredict ? len : Elem<Ein>::kChunk,
                                           kPredict && cc.i > 0 && row_inf,
                                           kPredict ? &had_inf : nullptr);
            if (kPredict && cc.i == 0) row_inf = had_inf;
            if (lane == 0) records[b * kFbMaxChunks + tk.g] = rec;
            if (cc.i == cc.cnt - 1) {
                // This warp's last chunk of the row.  With the backward, every
                // warp waits for the fold anyway, so the last warp to get here
                // folds.  Forward only, nobody waits for it, and the folding
                // warp starts its next row late: the row's folding warp (see
                // n_fold) folds it once the others' records are in; with 38
                // chunks that is warp 12, whose row has one chunk less.
                __syncwarp();
                bool fold_now;
                if constexpr (kBwd) {
                    int arrived = 0;
                    if (lane == 0) {
                        __threadfence_block();
                        arrived = atomicAdd(&counter[b], 1);
                    }
                    arrived = __shfl_sync(0xFFFFFFFFu, arrived, 0);
                    fold_now = arrived == active - 1;
                } else if (kOwnFolder || warp != active - 1 - (int)(tk.r % n_fold)) {
                    if (lane == 0) mbar_arrive(&recs[b]);  // release: this warp's records
                    fold_now = false;
                } else {
                    bool ok = active == 1 ||
                              mbar_wait_bounded(&recs[b], (uint32_t)((tk.r >> 1) & 1), kWaitLimitNs);
                    ok = __all_sync(0xFFFFFFFFu, ok);
                    if (!ok) {
                        failed = true;
                        break;
                    }
                    fold_now = true;
                }
                if (fold_now) {
                    // fold_row's steps, written out in place: as a call they
                    // measured 0.24% slower in the single pass and 1.1% in the
                    // forward.  The tests compare the two paths bit for bit.
                    __threadfence_block();
                    // Label, weight and z_y first (for rows past the cache
                    // the z_y load then runs under the fold's arithmetic).
                    const int64_t t = tk.t;
                    const bool cached = tk.r < kFbRowCache;
                    const int64_t y = cached ? lab_s[tk.r] : (labels ? labels[t] : ignore_index);
                    const float w = cached ? wt_s[tk.r] : (weights ? weights[t] : 1.f);
                    const int64_t yl = kShard ? y - label_offset : y;  // the label's column here
                    const bool y_in = y != ignore_index && yl >= 0 && yl < V;
                    float zy = 0.f;
                    if (lane == 0 && y_in)
                        zy = cached ? zy_s[tk.r] : Elem<Ein>::to_float(logits[t * ld + yl]);
                    const float3 st = fold_row_warp(records + b * kFbMaxChunks, plan, lane);
                    if (kShard && lane == 0) {
                        shard_out[t] = make_float4(st.x, st.y, st.z, zy);
                        mbar_arrive(&ready[b]);
                    } else if (lane == 0) {
                        counter[b] = 0;
                        const float M = st.x, S = st.y, U = st.z;
                        // First what pass 2 waits for -- ln S, the row's mode and
                        // its gradient constants -- then publish; the entropy
                        // (a division) and the global stores come after.
                        const bool empty = !(M > -INFINITY);
                        const bool bad = !empty && y != ignore_index && (y < 0 || y >= V);
                        const float lnS = empty ? NAN : logf(S);
                        RowInfo nr;
                        nr.mode = (y == ignore_index || w == 0.f) ? 0 : (empty || bad) ? 1 : 2;
                        nr.gr = nr.mode == 2 ? grad_row(M, lnS, w) : GradRow{0.f, 0.f, 0.f, 0.f};
                        nr.y = y;
                        nr.zy = zy;
                        info[b] = nr;
                        mbar_arrive(&ready[b]);  // release: records, info visible to waiters
                        float H, lp;
                        if (empty) {
                            H = NAN;
                            lp = NAN;
                        } else {
                            H = lnS - U / S;
                            if (y == ignore_index) {
                                lp = 0.f;
                            } else if (bad) {
                                lp = NAN;
                                H = NAN;
                            } else {
                                lp = (zy - M) - lnS;
                            }
                        }
                        if (logprob) logprob[t] = lp;
                        if (entropy) entropy[t] = H;
                        if (rowstats) reinterpret_cast<float2*>(rowstats)[t] = make_float2(M, lnS);
                        const int err = (empty ? PSTAT_DEV_EMPTY_ROW : 0) | (bad ? PSTAT_DEV_BAD_LABEL : 0);
                        if (err && dev_error) atomicOr(dev_error, err);
                    }
                }
                __syncwarp();
            }
        } else if constexpr (kBwd) {
            // dlogits of this chunk: columns [start, start + len) of row t
            Eout* dst = out + tk.t * ld_out + start;
            const int64_t y = ri.y;
            const bool vec_ok = ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0) &&
                                (len % kVec == 0);
            if (ri.mode == 2) {
                const bool has_y = y >= start && y < start + len;
                if (vec_ok && nvec == 32 * kVecPerLane) {
                    // full aligned chunk: no per-vector tests
                    Eout* d = dst + lane * kVec;
#pragma unroll
                    for (int jj = 0; jj < kVecPerLane; ++jj) {
                        float x[kVec], gv[kVec];
                        unpack_vec<Ein>(q[jj], x);
                        grad_vec_nolabel<kVec>(x, ri, gv);
                        OutVec<Eout>::template store<kVec>(d + 32 * kVec * jj, gv);
                    }
                    if (has_y && (int)(((y - start) / kVec) & 31) == lane) {
                        // The lane that stored the label's vector rewrites the label
                        // column with w (1 - p_y), e_y from the same arithmetic.
                        float x8[8], e8[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) x8[e] = ri.zy;
                        exp8(x8, ri.gr.m2, e8);
                        dst[y - start] = OutVec<Eout>::one(grad_label(e8[0], ri.gr));
                    }
                } else {
#pragma unroll
                    for (int jj = 0; jj < kVecPerLane; ++jj) {
                        const int k = lane + 32 * jj;
                        if (k >= nvec) break;
                        float x[kVec], gv[kVec];
                        unpack_vec<Ein>(q[jj], x);
                        grad_vec<kVec>(x, ri, start + (int64_t)k * kVec, y, gv);
                        if (vec_ok) {
                            OutVec<Eout>::template store<kVec>(dst + (int64_t)k * kVec, gv);
                        } else {
#pragma unroll
                            for (int e = 0; e < kVec; ++e)
                                if (k * kVec + e < len)
                                    dst[(int64_t)k * kVec + e] = OutVec<Eout>::one(gv[e]);
                        }
                    }
                }
            } else {
                const float fill = (ri.mode == 0) ? 0.f : NAN;
                float gv[kVec];
#pragma unroll
                for (int e = 0; e < kVec; ++e) gv[e] = fill;
                for (int k = lane; k < nvec; k += 32) {
                    if (vec_ok) {
                        OutVec<Eout>::template store<kVec>(dst + (int64_t)k * kVec, gv);
                    } else {
                        for (int e = 0; e < kVec; ++e)
                            if (k * kVec + e < len) dst[(int64_t)k * kVec + e] = OutVec<Eout>::one(fill);
                    }
                }
            }
        }
        if (!hold) ++pc;
        advance(cc);
    }
    if (failed) {
        if (lane == 0 && dev_error) atomicOr(dev_error, PSTAT_DEV_TIMEOUT);
        // Drain copies still in flight into this CTA's shared memory before leaving
        // (held positions had no copy).
        for (int64_t p = pc; p < pi && !done(cc);) {
            if (!held(cc)) {
                if (!in_slot(cc) && task_of(cc).bulk) {
                    const int slot = (int)(p % kFbStages);
                    mbar_wait_bounded(&bars[slot], (phase >> slot) & 1u, kWaitLimitNs);
                    phase ^= 1u << slot;
                }
                ++p;
            }
            advance(cc);
        }
    }
}

template <typename Ein, typename Eout, bool kBwd, bool kShard = false, bool kShards = false,
          bool kOwnFolder = false>
cudaError_t launch_fused_one(const Ein* logits, int64_t T, int64_t V, int64_t ld,
                           const ShardPlan& plan, const int64_t* labels, int64_t ignore_index,
                           const float* weights, float* logprob, float* entropy, float* rowstats,
                           Eout* out, int64_t ld_out, int* dev_error, const DeviceInfo& dev,
                           cudaStream_t stream, float4* shard_out = nullptr,
                           int64_t label_offset = 0) {
    static ContextSeen configured;
    const cudaError_t e = ensure_smem_optin(
        reinterpret_cast<const void*>(fwdbwd_kernel<Ein, Eout, kBwd, kShard, kShards, kOwnFolder>),
        (int)kFusedSmem,
        configured);
    if (e != cudaSuccess) return e;
    int64_t cap = dev.sm_count;
    if constexpr (kBwd && sizeof(Ein) == 4) {
        // Every CTA holds its current row in L2 between the two passes.  fp32
        // rows of 608 KB (V = 151,936) on all 152 SMs, 92 MB of the 135.5 MB
        // L2, missed it in pass 2 (DRAM reads 1.33x the logits).  A sweep of
        // the grid at T = 8192 put the best near three quarters of the SMs
        // (114 CTAs: 1.63 against 1.87 ms).  bf16 rows carry twice the
        // elements per byte and wanted more SMs (304 KB rows: all 152; 600 KB:
        // 136, 5% ahead of 152), so they keep every SM.
        const int64_t row_bytes = V * (int64_t)sizeof(Ein);
        if (2 * row_bytes * dev.sm_count > (int64_t)dev.l2_bytes) cap = dev.sm_count * 3 / 4;
    }
    const int64_t grid = T < cap ? T : cap;
    fwdbwd_kernel<Ein, Eout, kBwd, kShard, kShards, kOwnFolder>
        <<<(unsigned)grid, (kFbWarps + (kOwnFolder ? 1 : 0)) * 32, kFusedSmem, stream>>>(
        logits, T, V, ld, plan, labels, ignore_index, weights, logprob, entropy, rowstats, out,
        ld_out, shard_out, label_offset, dev_error);
    return cudaGetLastError();
}

template <typename Ein, typename Eout, bool kBwd, bool kShard = false>
cudaError_t launch_fused_t(const Ein* logits, int64_t T, int64_t V, int64_t ld,
                           const ShardPlan& plan, const int64_t* labels, int64_t ignore_index,
                           const float* weights, float* logprob, float* entropy, float* rowstats,
                           Eout* out, int64_t ld_out, int* dev_error, const DeviceInfo& dev,
                           cudaStream_t stream, float4* shard_out = nullptr,
                           int64_t label_offset = 0) {
    if constexpr (kBwd) {
        if (plan.n_shards > 1)
            return launch_fused_one<Ein, Eout, kBwd, kShard, true>(
                logits, T, V, ld, plan, labels, ignore_index, weights, logprob, entropy, rowstats,
                out, ld_out, dev_error, dev, stream, shard_out, label_offset);
    } else {
        // A warp of its own folds the rows when every chunk-owning warp holds
        // as many chunks of a row; otherwise the warps with one chunk less do.
        if (plan.n_chunks < kFbWarps || plan.n_chunks % kFbWarps == 0)
            return launch_fused_one<Ein, Eout, kBwd, kShard, false, true>(
                logits, T, V, ld, plan, labels, ignore_index, weights, logprob, entropy, rowstats,
                out, ld_out, dev_error, dev, stream, shard_out, label_offset);
    }
    return launch_fused_one<Ein, Eout, kBwd, kShard, false>(
        logits, T, V, ld, plan, labels, ignore_index, weights, logprob, entropy, rowstats, out,
        ld_out, dev_error, dev, stream, shard_out, label_offset);
}

}  // namespace

int forward_rows_max_chunks() { return kFbMaxChunks; }

cudaError_t launch_forward_rows(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                int64_t ld, const ShardPlan& plan, const int64_t* labels,
                                int64_t ignore_index, float* logprob, float* entropy,
                                float* rowstats, int* dev_error, const DeviceInfo& dev,
                                cudaStream_t stream, float4* shard_out, int64_t label_offset) {
    if (plan.n_chunks > kFbMaxChunks) return cudaErrorInvalidValue;
    const uint16_t* zb = static_cast<const uint16_t*>(logits);
    const float* zf = static_cast<const float*>(logits);
    if (shard_out && dt == PSTAT_BF16)
        return launch_fused_t<uint16_t, float, false, true>(
            zb, T, V, ld, plan, labels, ignore_index, nullptr, logprob, entropy, rowstats, nullptr,
            0, dev_error, dev, stream, shard_out, label_offset);
    if (shard_out)
        return launch_fused_t<float, float, false, true>(
            zf, T, V, ld, plan, labels, ignore_index, nullptr, logprob, entropy, rowstats, nullptr,
            0, dev_error, dev, stream, shard_out, label_offset);
    if (dt == PSTAT_BF16)
        return launch_fused_t<uint16_t, float, false>(zb, T, V, ld, plan, labels, ignore_index,
                                                      nullptr, logprob, entropy, rowstats, nullptr,
                                                      0, dev_error, dev, stream);
    return launch_fused_t<float, float, false>(zf, T, V, ld, plan, labels, ignore_index, nullptr,
                                               logprob, entropy, rowstats, nullptr, 0, dev_error,
                                               dev, stream);
}

}  // namespace pstat

using namespace pstat;

extern "C" int pstat_forward_backward(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                      int64_t ld, const int64_t* labels, int64_t ignore_index,
                                      const float* weights, const int64_t* shard_bounds,
                                      int n_shards, float* out_logprob, float* out_entropy,
                                      float* out_rowstats, void* out_dlogits, pstat_dtype out_dt,
                                      int64_t ld_out, int* dev_error, pstat_stream_t stream) {
    if ((dt != PSTAT_F32 && dt != PSTAT_BF16) || (out_dt != PSTAT_F32 && out_dt != PSTAT_BF16))
        return PSTAT_ERR_DTYPE;
    if (dt == PSTAT_BF16 && out_dt == PSTAT_F32) return PSTAT_ERR_DTYPE;
    if (T < 0 || V < 1 || ld < V || ld_out < V) return PSTAT_ERR_SHAPE;
    ShardPlan plan;
    int rc = make_plan(V, dt == PSTAT_BF16 ? PSTAT_CHUNK_BF16 : PSTAT_CHUNK_F32, shard_bounds,
                       n_shards, &plan);
    if (rc != PSTAT_OK) return rc;
    if (plan.n_chunks > kFbMaxChunks) return PSTAT_ERR_SHAPE;
    if (T == 0) return PSTAT_OK;
    if (!logits || !out_dlogits) return PSTAT_ERR_NULLPTR;
    const size_t ein = dt == PSTAT_BF16 ? 2 : 4, eout = out_dt == PSTAT_BF16 ? 2 : 4;
    if ((reinterpret_cast<uintptr_t>(logits) % ein) != 0 ||
        (reinterpret_cast<uintptr_t>(out_dlogits) % eout) != 0)
        return PSTAT_ERR_ALIGN;
    if ((out_rowstats && (reinterpret_cast<uintptr_t>(out_rowstats) & 7u)) ||
        (labels && (reinterpret_cast<uintptr_t>(labels) & 7u)) ||
        (weights && (reinterpret_cast<uintptr_t>(weights) & 3u)))
        return PSTAT_ERR_ALIGN;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dt == PSTAT_BF16)
        e = launch_fused_t<uint16_t, uint16_t, true>(static_cast<const uint16_t*>(logits), T, V,
                           ld, plan, labels, ignore_index, weights, out_logprob, out_entropy, out_rowstats,
                           static_cast<uint16_t*>(out_dlogits), ld_out, dev_error, dev, st);
    else if (out_dt == PSTAT_BF16)
        e = launch_fused_t<float, uint16_t, true>(static_cast<const float*>(logits), T, V, ld,
                           plan, labels, ignore_index, weights, out_logprob, out_entropy, out_rowstats,
                           static_cast<uint16_t*>(out_dlogits), ld_out, dev_error, dev, st);
    else
        e = launch_fused_t<float, float, true>(static_cast<const float*>(logits), T, V, ld,
                           plan, labels, ignore_index, weights, out_logprob, out_entropy, out_rowstats,
                           static_cast<float*>(out_dlogits), ld_out, dev_error, dev, st);
    return e == cudaSuccess ? PSTAT_OK : PSTAT_ERR_CUDA;
}
