// internal.h -- declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "pstat.h"

namespace pstat {

// Fixed chunk plan of one row, identical for every row of a call: the chunks
// restart at every shard start (so a shard's statistics are what a tensor-
// parallel rank holding [b_s, b_{s+1}) would compute locally).
struct ShardPlan {
    int n_shards;
    int n_chunks;                            // chunks per row
    int chunk;                               // chunk length in elements
    int cum[PSTAT_MAX_SHARDS + 1];           // first chunk index of each shard
    int64_t bounds[PSTAT_MAX_SHARDS + 1];    // shard column bounds
};

// Builds the plan; returns PSTAT_OK or PSTAT_ERR_SHARDS.
int make_plan(int64_t V, int chunk, const int64_t* bounds, int n_shards, ShardPlan* plan);

constexpr size_t kChunkRecordBytes = 16;  // (m, s, u, unused) fp32

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout of pstat_forward / pstat_backward.
struct StatsWorkspace {
    size_t chunk_stats_off;  // [T, n_chunks] float4
    size_t rowstats_off;     // [T, 2] float
    size_t total;
};
StatsWorkspace stats_workspace_layout(int64_t T, const ShardPlan& plan);

// Device properties cached per device.
struct DeviceInfo {
    int sm_count;
    int cc_major, cc_minor;
    int max_smem_optin;
    int l2_bytes;
};
int device_info(DeviceInfo* info);  // PSTAT_OK / PSTAT_ERR_CUDA / PSTAT_ERR_UNSUPPORTED

// Per-context set-up.  A kernel's shared-memory opt-in and the device address
// of a __device__ array belong to the module loaded in one CUDA context; after
// cudaDeviceReset the module is loaded again into a new context, where the
// attribute is back at its default and the array may sit elsewhere.  Caches of
// such set-up are therefore keyed on the context's process-unique id
// (cuCtxGetId), never on the device index alone.
constexpr int kMaxDevices = 64;

// Id of the context current on this thread; 0 when none is current yet or
// the CUDA driver cannot report it (callers then redo their set-up every time).
uint64_t current_context_id();

// For each device, the id of the context in which a one-time set-up last ran.
struct ContextSeen {
    std::atomic<uint64_t> id[kMaxDevices];
};

// cudaFuncSetAttribute(func, MaxDynamicSharedMemorySize, bytes), run once per
// device and context.
cudaError_t ensure_smem_optin(const void* func, int bytes, ContextSeen& seen);

// Kernel launchers (stats_kernels.cu).  They assume validated arguments.
cudaError_t launch_chunk_stats(const void* logits, pstat_dtype dt, int64_t T, int64_t ld,
                               const ShardPlan& plan, float4* chunk_stats, int* dev_error,
                               const DeviceInfo& dev, cudaStream_t stream);
cudaError_t launch_combine(const float4* chunk_stats, const ShardPlan& plan, const void* logits,
                           pstat_dtype dt, int64_t T, int64_t V, int64_t ld,
                           const int64_t* labels, int64_t ignore_index, const float* target,
                           float* logprob, float* entropy, float* rowstats, int* dev_error,
                           cudaStream_t stream);
cudaError_t launch_backward(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                            int64_t ld, const int64_t* labels, int64_t ignore_index,
                            const float* weights, const float* rowstats, void* out,
                            pstat_dtype out_dt, int64_t ld_out, int* dev_error,
                            const DeviceInfo& dev, cudaStream_t stream,
                            int64_t label_offset = 0, int64_t v_total = -1);

cudaError_t launch_logsoftmax(const void* logits, pstat_dtype dt, int64_t T, int64_t V, int64_t ld,
                              const float* rowstats, void* out, pstat_dtype out_dt, int64_t ld_out,
                              int* dev_error, cudaStream_t stream);

// The forward in one kernel (fused.cu): the single-pass kernel's first pass,
// chunk records in shared memory, each row folded by the warp that finishes
// it; the same records, fold and outputs as launch_chunk_stats + launch_combine,
// bit for bit.  Plans with more than forward_rows_max_chunks() chunks per row
// return cudaErrorInvalidValue without launching.  With shard_out the kernel
// writes each row's (M, S, U, z_y) for a vocabulary shard instead of the row
// outputs (labels numbered from label_offset; z_y = 0 off the shard).
int forward_rows_max_chunks();
cudaError_t launch_forward_rows(const void* logits, pstat_dtype dt, int64_t T, int64_t V,
                                int64_t ld, const ShardPlan& plan, const int64_t* labels,
                                int64_t ignore_index, float* logprob, float* entropy,
                                float* rowstats, int* dev_error, const DeviceInfo& dev,
                                cudaStream_t stream, float4* shard_out = nullptr,
                                int64_t label_offset = 0);

}  // namespace pstat
