// pstat_api.cu -- the extern "C" entry points of libpstat.so: argument
// checks, workspace layout and kernel launches on the caller's stream.
// Contracts are documented in include/pstat.h.
#include <cuda.h>  // CUcontext, CUresult (types only; the CUDA driver is reached by entry point)
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "internal.h"

namespace pstat {

namespace {
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

void* driver_entry(const char* name) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return p;
}
}  // namespace

uint64_t current_context_id() {
    static std::once_flag once;
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    std::call_once(once, [] {
        get_current = reinterpret_cast<CtxGetCurrentFn>(driver_entry("cuCtxGetCurrent"));
        get_id = reinterpret_cast<CtxGetIdFn>(driver_entry("cuCtxGetId"));
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
    unsigned long long id = 0;
    if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return (uint64_t)id;
}

cudaError_t ensure_smem_optin(const void* func, int bytes, ContextSeen& seen) {
    int d = 0;
    const cudaError_t ge = cudaGetDevice(&d);
    if (ge != cudaSuccess) return ge;
    const bool slot = d >= 0 && d < kMaxDevices;
    const uint64_t id = current_context_id();
    if (slot && id != 0 && seen.id[d].load(std::memory_order_acquire) == id) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    // The call above has made the device's primary context current if it was not.
    const uint64_t now = current_context_id();
    if (slot && now != 0) seen.id[d].store(now, std::memory_order_release);
    return cudaSuccess;
}

int make_plan(int64_t V, int chunk, const int64_t* bounds, int n_shards, ShardPlan* plan) {
    if (bounds == nullptr) {
        if (n_shards != 1 && n_shards != 0) return PSTAT_ERR_SHARDS;
        n_shards = 1;
    }
    if (n_shards < 1 || n_shards > PSTAT_MAX_SHARDS) return PSTAT_ERR_SHARDS;
    plan->n_shards = n_shards;
    plan->chunk = chunk;
    int64_t total = 0;
    plan->cum[0] = 0;
    for (int s = 0; s <= n_shards; ++s) {
        const int64_t b = bounds ? bounds[s] : (s == 0 ? 0 : V);
        plan->bounds[s] = b;
        if (s == 0 && b != 0) return PSTAT_ERR_SHARDS;
        if (s > 0) {
            if (b <= plan->bounds[s - 1]) return PSTAT_ERR_SHARDS;
            total += (b - plan->bounds[s - 1] + chunk - 1) / chunk;
            if (total > (1 << 24)) return PSTAT_ERR_SHAPE;
            plan->cum[s] = (int)total;
        }
    }
    if (plan->bounds[n_shards] != V) return PSTAT_ERR_SHARDS;
    for (int s = n_shards + 1; s <= PSTAT_MAX_SHARDS; ++s) {
        plan->cum[s] = (int)total;
        plan->bounds[s] = V;
    }
    plan->n_chunks = (int)total;
    return PSTAT_OK;
}

StatsWorkspace stats_workspace_layout(int64_t T, const ShardPlan& plan) {
    StatsWorkspace w;
    w.chunk_stats_off = 0;
    w.rowstats_off = align_up((size_t)T * plan.n_chunks * kChunkRecordBytes, 256);
    w.total = align_up(w.rowstats_off + (size_t)T * 2 * sizeof(float), 256);
    return w;
}

int device_info(DeviceInfo* info) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    static bool have[64] = {};
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess) return PSTAT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (d >= 64 || !have[d]) {
        DeviceInfo di;
        if (cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, d) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, d) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&di.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                   d) != cudaSuccess ||
            cudaDeviceGetAttribute(&di.l2_bytes, cudaDevAttrL2CacheSize, d) != cudaSuccess)
            return PSTAT_ERR_CUDA;
        if (d < 64) {
            cache[d] = di;
            have[d] = true;
        } else {
            *info = di;
        }
    }
    if (d < 64) *info = cache[d];
    // The kernels are built for sm_103a only.
    if (info->cc_major != 10 || info->cc_minor != 3) return PSTAT_ERR_UNSUPPORTED;
    return PSTAT_OK;
}

static int chunk_for(pstat_dtype dt) { return dt == PSTAT_BF16 ? PSTAT_CHUNK_BF16 : PSTAT_CHUNK_F32; }
static size_t elem_size(pstat_dtype dt) { return dt == PSTAT_BF16 ? 2 : 4; }
static bool valid_dtype(int dt) { return dt == PSTAT_F32 || dt == PSTAT_BF16; }

}  // namespace pstat

using namespace pstat;

extern "C" {

const char* pstat_status_string(int code) {
    switch (code) {
        case PSTAT_OK: return "ok";
        case PSTAT_ERR_NULLPTR: return "a required pointer is NULL";
        case PSTAT_ERR_SHAPE: return "invalid shape (T, V, ld, d)";
        case PSTAT_ERR_SHARDS: return "invalid shard bounds";
        case PSTAT_ERR_DTYPE: return "unsupported dtype";
        case PSTAT_ERR_ALIGN: return "pointer not aligned as required";
        case PSTAT_ERR_WORKSPACE: return "workspace missing or too small";
        case PSTAT_ERR_CUDA: return "CUDA runtime error";
        case PSTAT_ERR_UNSUPPORTED: return "device is not sm_103 (GB300)";
        default: return "unknown status";
    }
}

int pstat_version(void) { return 10000; }

int pstat_workspace_size(int64_t T, int64_t V, pstat_dtype dt, const int64_t* shard_bounds,
                         int n_shards, size_t* bytes) {
    if (!bytes) return PSTAT_ERR_NULLPTR;
    if (!valid_dtype(dt)) return PSTAT_ERR_DTYPE;
    if (T < 0 || V < 1) return PSTAT_ERR_SHAPE;
    ShardPlan plan;
    const int rc = make_plan(V, chunk_for(dt), shard_bounds, n_shards, &plan);
    if (rc != PSTAT_OK) return rc;
    *bytes = stats_workspace_layout(T, plan).total;
    return PSTAT_OK;
}

int pstat_forward(const void* logits, pstat_dtype dt, int64_t T, int64_t V, int64_t ld,
                  const int64_t* labels, int64_t ignore_index, const int64_t* shard_bounds,
                  int n_shards, float* out_logprob, float* out_entropy, float* out_rowstats,
                  void* workspace, size_t ws_bytes, int* dev_error, pstat_stream_t stream) {
    if (!valid_dtype(dt)) return PSTAT_ERR_DTYPE;
    if (T < 0 || V < 1 || ld < V) return PSTAT_ERR_SHAPE;
    ShardPlan plan;
    int rc = make_plan(V, chunk_for(dt), shard_bounds, n_shards, &plan);
    if (rc != PSTAT_OK) return rc;
    if (T == 0) return PSTAT_OK;
    if (!logits) return PSTAT_ERR_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(logits) % elem_size(dt)) != 0) return PSTAT_ERR_ALIGN;
    if ((out_rowstats && (reinterpret_cast<uintptr_t>(out_rowstats) & 7u)) ||
        (labels && (reinterpret_cast<uintptr_t>(labels) & 7u)))
        return PSTAT_ERR_ALIGN;
    // The one-kernel path keeps the chunk records in shared memory and needs
    // no workspace; larger plans need one.
    const bool one_kernel = plan.n_chunks <= forward_rows_max_chunks();
    const StatsWorkspace wl = stats_workspace_layout(T, plan);
    if (!one_kernel) {
        if (!workspace || ws_bytes < wl.total) return PSTAT_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return PSTAT_ERR_ALIGN;
    }
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (one_kernel) {
        return launch_forward_rows(logits, dt, T, V, ld, plan, labels, ignore_index, out_logprob,
                                   out_entropy, out_rowstats, dev_error, dev, st) == cudaSuccess
                   ? PSTAT_OK
                   : PSTAT_ERR_CUDA;
    }
    float4* cs = reinterpret_cast<float4*>(static_cast<char*>(workspace) + wl.chunk_stats_off);
    if (launch_chunk_stats(logits, dt, T, ld, plan, cs, dev_error, dev, st) != cudaSuccess)
        return PSTAT_ERR_CUDA;
    if (launch_combine(cs, plan, logits, dt, T, V, ld, labels, ignore_index, nullptr,
                       out_logprob, out_entropy, out_rowstats, dev_error, st) != cudaSuccess)
        return PSTAT_ERR_CUDA;
    return PSTAT_OK;
}

int pstat_backward(const void* logits, pstat_dtype dt, int64_t T, int64_t V, int64_t ld,
                   const int64_t* labels, int64_t ignore_index, const float* weights,
                   const float* rowstats, const int64_t* shard_bounds, int n_shards,
                   void* out_dlogits, pstat_dtype out_dt, int64_t ld_out, void* workspace,
                   size_t ws_bytes, int* dev_error, pstat_stream_t stream) {
    if (!valid_dtype(dt) || !valid_dtype(out_dt)) return PSTAT_ERR_DTYPE;
    if (dt == PSTAT_BF16 && out_dt == PSTAT_F32) return PSTAT_ERR_DTYPE;
    if (T < 0 || V < 1 || ld < V || ld_out < V) return PSTAT_ERR_SHAPE;
    ShardPlan plan;
    int rc = make_plan(V, chunk_for(dt), shard_bounds, n_shards, &plan);
    if (rc != PSTAT_OK) return rc;
    if (T == 0) return PSTAT_OK;
    if (!logits || !out_dlogits) return PSTAT_ERR_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(logits) % elem_size(dt)) != 0 ||
        (reinterpret_cast<uintptr_t>(out_dlogits) % elem_size(out_dt)) != 0)
        return PSTAT_ERR_ALIGN;
    if ((rowstats && (reinterpret_cast<uintptr_t>(rowstats) & 7u)) ||
        (labels && (reinterpret_cast<uintptr_t>(labels) & 7u)) ||
        (weights && (reinterpret_cast<uintptr_t>(weights) & 3u)))
        return PSTAT_ERR_ALIGN;
    const StatsWorkspace wl = stats_workspace_layout(T, plan);
    if (rowstats == nullptr) {
        if (!workspace || ws_bytes < wl.total) return PSTAT_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return PSTAT_ERR_ALIGN;
    }
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const float* rs = rowstats;
    if (rs == nullptr) {
        char* ws = static_cast<char*>(workspace);
        float4* cs = reinterpret_cast<float4*>(ws + wl.chunk_stats_off);
        float* rws = reinterpret_cast<float*>(ws + wl.rowstats_off);
        if (plan.n_chunks <= forward_rows_max_chunks()) {
            if (launch_forward_rows(logits, dt, T, V, ld, plan, labels, ignore_index, nullptr,
                                    nullptr, rws, dev_error, dev, st) != cudaSuccess)
                return PSTAT_ERR_CUDA;
        } else {
            if (launch_chunk_stats(logits, dt, T, ld, plan, cs, dev_error, dev, st) != cudaSuccess)
                return PSTAT_ERR_CUDA;
            if (launch_combine(cs, plan, logits, dt, T, V, ld, labels, ignore_index, nullptr,
                               nullptr, nullptr, rws, dev_error, st) != cudaSuccess)
                return PSTAT_ERR_CUDA;
        }
        rs = rws;
    }
    if (launch_backward(logits, dt, T, V, ld, labels, ignore_index, weights, rs, out_dlogits,
                        out_dt, ld_out, dev_error, dev, st) != cudaSuccess)
        return PSTAT_ERR_CUDA;
    return PSTAT_OK;
}

int pstat_log_softmax(const void* logits, pstat_dtype dt, int64_t T, int64_t V, int64_t ld,
                      const float* rowstats, const int64_t* shard_bounds, int n_shards,
                      void* out, pstat_dtype out_dt, int64_t ld_out, void* workspace,
                      size_t ws_bytes, int* dev_error, pstat_stream_t stream) {
    if (!valid_dtype(dt) || !valid_dtype(out_dt)) return PSTAT_ERR_DTYPE;
    if (T < 0 || V < 1 || ld < V || ld_out < V) return PSTAT_ERR_SHAPE;
    ShardPlan plan;
    int rc = make_plan(V, chunk_for(dt), shard_bounds, n_shards, &plan);
    if (rc != PSTAT_OK) return rc;
    if (T == 0) return PSTAT_OK;
    if (!logits || !out) return PSTAT_ERR_NULLPTR;
    if ((reinterpret_cast<uintptr_t>(logits) % elem_size(dt)) != 0 ||
        (reinterpret_cast<uintptr_t>(out) % elem_size(out_dt)) != 0 ||
        (rowstats && (reinterpret_cast<uintptr_t>(rowstats) & 7u)))
        return PSTAT_ERR_ALIGN;
    const StatsWorkspace wl = stats_workspace_layout(T, plan);
    if (rowstats == nullptr) {
        if (!workspace || ws_bytes < wl.total) return PSTAT_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0) return PSTAT_ERR_ALIGN;
    }
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    const float* rs = rowstats;
    if (rs == nullptr) {
        char* ws = static_cast<char*>(workspace);
        float4* cs = reinterpret_cast<float4*>(ws + wl.chunk_stats_off);
        float* rws = reinterpret_cast<float*>(ws + wl.rowstats_off);
        if (launch_chunk_stats(logits, dt, T, ld, plan, cs, dev_error, dev, st) != cudaSuccess)
            return PSTAT_ERR_CUDA;
        if (launch_combine(cs, plan, logits, dt, T, V, ld, nullptr, -1, nullptr, nullptr, nullptr,
                           rws, dev_error, st) != cudaSuccess)
            return PSTAT_ERR_CUDA;
        rs = rws;
    }
    if (launch_logsoftmax(logits, dt, T, V, ld, rs, out, out_dt, ld_out, dev_error, st) !=
        cudaSuccess)
        return PSTAT_ERR_CUDA;
    return PSTAT_OK;
}

}  // extern "C"
