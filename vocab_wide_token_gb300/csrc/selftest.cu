// selftest.cu -- pstat_selftest_wait_timeout: the bounded wait that every
// kernel of this library puts on its mbarriers, run against a barrier that
// nothing ever arrives at.  The wait gives up after the limit, the kernel
// sets PSTAT_DEV_TIMEOUT and returns; no copy is in flight, so nothing is
// left to drain and the context stays usable.
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace pstat {
namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, int* dev_error) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    // Phase 0 completes only after one arrival, and none comes.
    if (!mbar_wait_bounded(&bar, 0, limit_ns) && dev_error)
        atomicOr(dev_error, PSTAT_DEV_TIMEOUT);
}

}  // namespace
}  // namespace pstat

using namespace pstat;

extern "C" int pstat_selftest_wait_timeout(uint64_t limit_ns, int* dev_error,
                                           pstat_stream_t stream) {
    if (!dev_error) return PSTAT_ERR_NULLPTR;
    if (limit_ns > 1000000000ull) return PSTAT_ERR_SHAPE;
    DeviceInfo dev;
    const int rc = device_info(&dev);
    if (rc != PSTAT_OK) return rc;
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns, dev_error);
    return cudaGetLastError() == cudaSuccess ? PSTAT_OK : PSTAT_ERR_CUDA;
}
