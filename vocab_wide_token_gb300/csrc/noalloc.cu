// noalloc.cu -- pstat_forward_noalloc: the forward statistics without a
// caller-supplied workspace and without any allocation.
//
// Who needs this: callers that are not allowed to allocate device memory at
// the point where they compute statistics.  cudaMalloc and cudaFree
// synchronise the whole device, so latency-critical loops avoid them; hosts
// that hand all device memory to their own pool (a serving runtime, a plug-in
// inside another framework, a process running under a fixed memory budget)
// forbid allocations outside that pool; and a plain C caller may simply have
// no allocator to hand.  Such a caller still owns its inputs and outputs, but
// it cannot provide the scratch that pstat_forward keeps its per-chunk
// statistics in.
//
// Instead, the scratch is a fixed array in device memory that belongs to
// this library (PSTAT_NOALLOC_SCRATCH_BYTES per GPU, held from the moment
// the library's module is loaded on that GPU until the process exits).  Host
// code cannot use the array's name as a device address, so the first call on
// each device looks the address up with cudaGetSymbolAddress while that
// device is current, and later calls reuse it.  The address belongs to the
// context the module was loaded in: after cudaDeviceReset the next call finds
// a new context (a new cuCtxGetId) and looks the address up again.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

// Per-(row, chunk) records of the chunk-statistics kernel.  Every record a
// call reads is written earlier in the same call, so nothing needs clearing
// between calls.
static __device__ __align__(256) float4 g_noalloc_scratch[PSTAT_NOALLOC_SCRATCH_BYTES / sizeof(float4)];

namespace pstat {
namespace {

struct ScratchAddress {
    uint64_t ctx_id;  // context the address was looked up in (0: none yet)
    float4* ptr;
};
std::mutex g_mu;
ScratchAddress g_scratch[kMaxDevices] = {};

// Device address of the scratch array in the current device's current
// context, looked up on the first call in that context.  Returns PSTAT_OK,
// PSTAT_ERR_CUDA or PSTAT_ERR_UNSUPPORTED.
int scratch_for_current_context(float4** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PSTAT_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PSTAT_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    const uint64_t id = current_context_id();
    if (id != 0 && g_scratch[dev].ctx_id == id) {
        *out = g_scratch[dev].ptr;
        return PSTAT_OK;
    }
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return PSTAT_ERR_CUDA;
    // The lookup has made the device's primary context current if it was not;
    // with no context id to key on, nothing is cached and the next call looks
    // the address up again.
    g_scratch[dev].ctx_id = current_context_id();
    g_scratch[dev].ptr = static_cast<float4*>(p);
    *out = g_scratch[dev].ptr;
    return PSTAT_OK;
}

}  // namespace
}  // namespace pstat

using namespace pstat;

extern "C" size_t pstat_noalloc_scratch_bytes(void) { return PSTAT_NOALLOC_SCRATCH_BYTES; }

extern "C" int pstat_forward_noalloc(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                     int64_t ld, const int64_t* labels, int64_t ignore_index,
                                     const int64_t* shard_bounds, int n_shards,
                                     float* out_logprob, float* out_entropy, float* out_rowstats,
                                     int* dev_error, pstat_stream_t stream) {
    if (dt != PSTAT_F32 && dt != PSTAT_BF16) return PSTAT_ERR_DTYPE;
    if (T < 0 || V < 1 || ld < V) return PSTAT_ERR_SHAPE;
    ShardPlan plan;
    int rc = make_plan(V, dt == PSTAT_BF16 ? PSTAT_CHUNK_BF16 : PSTAT_CHUNK_F32, shard_bounds,
                       n_shards, &plan);
    if (rc != PSTAT_OK) return rc;
    if (T == 0) return PSTAT_OK;
    if (!logits) return PSTAT_ERR_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(logits) % (dt == PSTAT_BF16 ? 2u : 4u)) != 0)
        return PSTAT_ERR_ALIGN;
    if ((out_rowstats && (reinterpret_cast<uintptr_t>(out_rowstats) & 7u)) ||
        (labels && (reinterpret_cast<uintptr_t>(labels) & 7u)))
        return PSTAT_ERR_ALIGN;
    // The whole problem must fit the fixed scratch: one 16-byte record per
    // row and chunk.
    const size_t need = (size_t)T * (size_t)plan.n_chunks * kChunkRecordBytes;
    if (need > (size_t)PSTAT_NOALLOC_SCRATCH_BYTES) return PSTAT_ERR_WORKSPACE;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    float4* cs = nullptr;
    rc = scratch_for_current_context(&cs);
    if (rc != PSTAT_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (launch_chunk_stats(logits, dt, T, ld, plan, cs, dev_error, dev, st) != cudaSuccess)
        return PSTAT_ERR_CUDA;
    if (launch_combine(cs, plan, logits, dt, T, V, ld, labels, ignore_index, nullptr,
                       out_logprob, out_entropy, out_rowstats, dev_error, st) != cudaSuccess)
        return PSTAT_ERR_CUDA;
    return PSTAT_OK;
}
