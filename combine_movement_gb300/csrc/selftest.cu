// selftest.cu -- exercises the failure path of the bounded waits on the GPU.
//
// Every mbarrier wait in the kernels gives up after a time limit and records
// EP_ERR_TIMEOUT in the caller's status word instead of spinning forever.
// ep_selftest_wait_timeout makes that happen on purpose, safely: one warp
// waits on the first of a ring of three freshly initialised mbarriers that
// nothing will ever complete, with a short limit, so the wait runs out and
// the status is written. It then drains the ring the way the copy kernels do
// after a timeout (one more bounded wait per stage that could still have a
// load in flight) and returns. The context stays usable.
#include <cuda_runtime.h>

#include "../../include/ep.h"
#include "ptx.cuh"

namespace {

constexpr int kRing = 3;

__global__ void wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar[kRing];
    const uint32_t b = ep::smem_u32(bar);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRing; ++s) ep::mbar_init(b + 8u * s, 1);  // no arrival will come
        ep::fence_mbar_init();
        if (!ep::mbar_wait_bounded(b, 0, limit_ns)) {
            ep::set_status(status, EP_ERR_TIMEOUT);
            ep::mbar_drain_bounded<kRing>(b, 0, kRing - 1, limit_ns);
        }
    }
}

}  // namespace

extern "C" ep_status_t ep_selftest_wait_timeout(int32_t* status, uint64_t limit_ns, void* stream) {
    if (status == nullptr || limit_ns == 0 || limit_ns > ep::kWaitLimitNs) return EP_ERR_INVALID;
    wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status, limit_ns);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}
