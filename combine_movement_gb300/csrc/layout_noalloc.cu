// layout_noalloc.cu -- ep_get_dispatch_layout_noalloc: the layout call for
// callers that cannot allocate device memory.
//
// Some callers have no way to hand this library a workspace. An inference
// server that reserved nearly all of HBM up front for weights and KV cache
// has nothing left for an extra cudaMalloc (it would fail, or fragment the
// reserved pool). A latency-critical pipeline cannot afford one either:
// cudaMalloc and cudaFree may synchronise the whole device and stall every
// stream that is in flight. For them the multi-tile layout's scratch (the
// barrier words and the per-(tile, expert) counts, kLayoutScratchBytes at
// most) lives in a file-scope __device__ array instead. Every GPU that loads
// the library holds that array until the process exits.
//
// Set-up: host code cannot pass the array's name to a kernel (on the host it
// is only a stand-in symbol, not a device address), so the first call on
// each device, with that device current, looks its address up with
// cudaGetSymbolAddress and caches it, together with the unique id of the
// CUDA context it was looked up in. A later call in another context of that
// device (after cudaDeviceReset, which destroys the primary context and
// with it the module that holds the array) looks it up again. Each lookup
// should therefore be made outside any stream capture: make the first call
// on a device, and the first one after a reset, before capturing.
//
// Sharing: every call uses the same array. Each call rewrites the counts it
// reads, and the barrier words it carries from call to call are valid from
// any starting value, so nothing has to start at zero; but calls that
// overlap on the GPU (different streams, or different host threads) race on
// the array and must be ordered by the caller.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/ep.h"
#include "kernels.cuh"

namespace {

constexpr size_t kLayoutScratchBytes = EP_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) int32_t g_layout_scratch[kLayoutScratchBytes / sizeof(int32_t)];

// Driver entry points for the current context's unique id (CUDA 12.0+),
// fetched through the runtime so the library links no driver library.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct ScratchCache {
    void* addr = nullptr;
    unsigned long long ctx_id = 0;
};

std::mutex g_scratch_mu;
ScratchCache g_scratch[kMaxDevices];
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
bool g_entry_points_tried = false;

// Unique id of the current CUDA context; 0 when no context is current yet.
// Returns false (and leaves the cache keyed by device alone) where the
// driver offers no context ids.
bool current_context_id(unsigned long long* out) {
    *out = 0;
    if (!g_entry_points_tried) {
        g_entry_points_tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
    }
    if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
        g_ctx_get_id(ctx, &id) == CUDA_SUCCESS)
        *out = id;
    return true;
}

// Device address of g_layout_scratch on the current device, looked up once
// per device and context.
ep_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EP_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchCache& c = g_scratch[dev];
    unsigned long long id = 0;
    const bool keyed = current_context_id(&id);
    if (c.addr == nullptr || (keyed && (id == 0 || id != c.ctx_id))) {
        // (the lookup makes the device's primary context current if it is
        // not yet, so the id taken after it is the context of the address)
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_layout_scratch) != cudaSuccess || p == nullptr)
            return EP_ERR_CUDA;
        c.addr = p;
        c.ctx_id = 0;
        if (keyed) current_context_id(&c.ctx_id);
    }
    *out = c.addr;
    return EP_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" ep_status_t ep_get_dispatch_layout_noalloc(const int64_t* topk_idx, int64_t T, int K,
                                                      int E, int32_t* counts, int32_t* offsets,
                                                      int32_t* slot, int32_t* status,
                                                      void* stream) {
    ep::ApiRange range("ep_get_dispatch_layout_noalloc");
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1) return EP_ERR_INVALID;
    if (E > EP_MAX_EXPERTS) return EP_ERR_UNSUPPORTED;
    if (T > ((int64_t{1} << 31) - 1) / K) return EP_ERR_UNSUPPORTED;  // T * K must fit int32
    if (counts == nullptr || offsets == nullptr) return EP_ERR_INVALID;
    if (T > 0 && (topk_idx == nullptr || slot == nullptr)) return EP_ERR_INVALID;
    if (!aligned(topk_idx, 8) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(slot, 4) ||
        !aligned(status, 4))
        return EP_ERR_INVALID;
    ep::LayoutPlan plan = ep::plan_layout(T * K, E);
    if (plan.workspace_bytes > kLayoutScratchBytes) return EP_ERR_UNSUPPORTED;
    // a table that one 16-CTA cluster can lay out needs no scratch at all
    // where the GPU holds one (and then shares nothing with other calls)
    if (plan.workspace_bytes > 0) (void)ep::plan_layout_wide_cluster(T * K, E, &plan);
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
