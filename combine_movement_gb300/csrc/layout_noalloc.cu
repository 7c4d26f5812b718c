// layout_noalloc.cu -- ep_get_dispatch_layout_noalloc: the layout call for
// callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace. An inference
// server that reserved nearly all of HBM up front for weights and KV cache
// has nothing left for an extra cudaMalloc (it would fail, or fragment the
// reserved pool). A latency-critical pipeline cannot afford one either:
// cudaMalloc and cudaFree may synchronise the whole device and stall every
// stream that is in flight. For them the multi-tile layout's scratch (the
// per-(expert, tile) counts, kLayoutScratchBytes at most) lives in a
// file-scope __device__ array instead. Every GPU that loads the library
// holds that array until the process exits.
//
// Set-up: host code cannot pass the array's name to a kernel (on the host it
// is only a stand-in symbol, not a device address), so the first call on
// each device, with that device current, looks its address up once with
// cudaGetSymbolAddress and caches it. That first call should therefore be
// made before any stream capture.
//
// Sharing: every call uses the same array. Each call rewrites the counts it
// reads, and the single generation word it carries from call to call is
// valid from any starting value, so nothing has to start at zero; but calls
// that overlap on the GPU (different streams, or different host threads)
// race on the array and must be ordered by the caller.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/ep.h"
#include "kernels.cuh"

namespace {

constexpr size_t kLayoutScratchBytes = EP_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) int32_t g_layout_scratch[kLayoutScratchBytes / sizeof(int32_t)];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_layout_scratch on the current device (looked up once
// per device).
ep_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess || p == nullptr)
            return EP_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return EP_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" ep_status_t ep_get_dispatch_layout_noalloc(const int64_t* topk_idx, int64_t T, int K,
                                                      int E, int32_t* counts, int32_t* offsets,
                                                      int32_t* slot, int32_t* status,
                                                      void* stream) {
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1) return EP_ERR_INVALID;
    if (E > EP_MAX_EXPERTS) return EP_ERR_UNSUPPORTED;
    if (T > ((int64_t{1} << 31) - 1) / K) return EP_ERR_UNSUPPORTED;  // T * K must fit int32
    if (counts == nullptr || offsets == nullptr) return EP_ERR_INVALID;
    if (T > 0 && (topk_idx == nullptr || slot == nullptr)) return EP_ERR_INVALID;
    if (!aligned(topk_idx, 8) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(slot, 4) ||
        !aligned(status, 4))
        return EP_ERR_INVALID;
    const ep::LayoutPlan plan = ep::plan_layout(T * K, E);
    if (plan.workspace_bytes > kLayoutScratchBytes) return EP_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (plan.workspace_bytes > 0) {
        const ep_status_t st = scratch_address(&scratch);
        if (st != EP_OK) return st;
    }
    const cudaError_t err =
        ep::launch_layout(topk_idx, T * K, E, counts, offsets, slot, scratch, plan, status,
                          static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}
