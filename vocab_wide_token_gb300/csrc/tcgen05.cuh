// tcgen05.cuh -- inline-PTX wrappers for the 5th-generation tensor cores
// (tcgen05.mma with accumulators in tensor memory), tensor-memory
// allocation and loads, and tiled TMA loads (cp.async.bulk.tensor).
#pragma once

#include <cuda.h>  // CUtensorMap (type only; no CUDA driver symbols are linked)

#include <cstdint>

#include "ptx.cuh"

namespace pstat {

// ---- tensor memory ------------------------------------------------------------
// Allocates `ncols` (power of two, 32..512) columns of tensor memory for this
// CTA; the whole warp executes it; the TMEM address lands in *smem_dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---- MMA ----------------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulation; issued by
// one thread.  `accumulate` = 0 overwrites D.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on `bar` when every tcgen05 operation this thread issued so
// far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, both K-major,
// shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4)                        // D format: f32
           | (1u << 7)                      // A format: bf16
           | (1u << 10)                     // B format: bf16
           | ((uint32_t)(N >> 3) << 17)     // N / 8
           | ((uint32_t)(M >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor for a K-major operand stored as rows of
// 128 bytes (64 bf16) with the 128-byte swizzle that TMA writes: 8-row
// groups of 1024 bytes follow each other (stride 1024 B).  The start address
// must lie in a 1024-byte aligned tile (advancing by 32 B per K step of 16
// stays inside the swizzle atom).
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t smem_addr) {
    return (uint64_t)((smem_addr >> 4) & 0x3FFFu)  // start address
           | ((uint64_t)1 << 16)                    // leading byte offset (unused here)
           | ((uint64_t)(1024 >> 4) << 32)          // stride byte offset
           | ((uint64_t)1 << 46)                    // descriptor version
           | ((uint64_t)2 << 61);                   // 128-byte swizzle
}

// Shared-memory matrix descriptor for an MN-major operand (its M or N index
// contiguous) written by TMA as boxes of 64 MN elements (128 bytes) x K rows
// with the 128-byte swizzle: one 8-row K group is a 1024-byte swizzle atom,
// the next K group follows at +1024 bytes (stride byte offset), and the next
// 64 MN elements sit `mn_stride` bytes further (leading byte offset, here the
// size of one box).  An MMA with K = 16 spans two K groups; successive K
// steps start 16 rows = 2048 bytes apart, so every start address is atom
// aligned.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t smem_addr, uint32_t mn_stride,
                                                        uint32_t k_stride = 1024) {
    return (uint64_t)((smem_addr >> 4) & 0x3FFFu)          // start address
           | ((uint64_t)((mn_stride >> 4) & 0x3FFFu) << 16)  // leading byte offset (MN)
           | ((uint64_t)((k_stride >> 4) & 0x3FFFu) << 32)   // stride byte offset (K)
           | ((uint64_t)1 << 46)                            // descriptor version
           | ((uint64_t)2 << 61);                           // 128-byte swizzle
}

// ---- tensor memory -> registers ------------------------------------------------
// Each thread of a warp reads 32 consecutive 32-bit columns of its own lane
// (the warp's lane quadrant is fixed by its warp index modulo 4).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---- tiled TMA ------------------------------------------------------------------
// 2-D tile load described by a tensor map; x is the innermost coordinate
// (must be a multiple of 8 bf16 elements = 16 bytes).
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// 4-D tile load (coordinates innermost first, x a multiple of 16 bytes).
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w),
        "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// 2-D tile store from shared memory (this thread's bulk async-group; x a
// multiple of 16 bytes, the source 128-byte aligned, laid out as the map's
// swizzle says).  The caller makes its shared-memory writes visible to the
// async proxy first (fence.proxy.async) and commits the group after.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y,
                                             const void* smem_src) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(smem_u32(smem_src))
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until at most N of this thread's bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait_group() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

}  // namespace pstat
