// kernels.cuh -- internal launch interface between the C ABI (ep_api.cu) and
// the kernels (layout.cu, dispatch.cu, combine.cu). Not part of the ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace ep {

// ---- layout ---------------------------------------------------------------

struct LayoutPlan {
    int warps;       // warps per block of the ranking kernel
    int rounds;      // 32-entry rounds per warp per tile
    int64_t tile;    // entries per tile = warps * 32 * rounds
    int num_tiles;   // 1 => single fused launch, no workspace
    size_t smem;     // dynamic shared memory of the ranking kernel
    size_t workspace_bytes;
};

LayoutPlan plan_layout(int64_t N, int E);

cudaError_t launch_layout(const int64_t* idx, int64_t N, int E, int32_t* counts,
                          int32_t* offsets, int32_t* slot, int32_t* tile_counts,
                          const LayoutPlan& plan, int32_t* status, cudaStream_t stream);

// ---- dispatch -------------------------------------------------------------

struct DispatchArgs {
    const uint8_t* x;
    int64_t T;
    uint32_t row_bytes;
    int K;
    const int32_t* slot;
    const float* topk_w;
    int64_t num_recv;
    uint8_t* recv_x;
    float* recv_w;
    int32_t* recv_src;
    int32_t* status;
    uint32_t chunk_bytes;  // bytes per row chunk (multiple of 16); last chunk may be shorter
    uint32_t n_chunks;     // chunks per row
    uint32_t stage_bytes;  // shared-memory bytes per ring stage (>= chunk_bytes)
};

cudaError_t launch_dispatch(const DispatchArgs& a, int num_sms, int smem_optin,
                            cudaStream_t stream);

// Largest ring stage (bytes, multiple of 16) dispatch can use on a device
// whose per-block shared-memory opt-in limit is `smem_optin`.
uint32_t dispatch_stage_capacity(int smem_optin);

// ---- combine --------------------------------------------------------------

struct CombineArgs {
    const uint8_t* expert_out;
    int64_t num_recv;
    const int32_t* slot;
    const float* topk_w;
    int64_t T;
    uint32_t row_bytes;
    int K;
    uint8_t* y;
    int32_t* status;
};

cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t stream);

// Combine with the expert rows staged through a per-warp bulk-copy ring
// (combine_tma.cu); K <= 8 only.
bool combine_tma_supported(int K);
cudaError_t launch_combine_tma(const CombineArgs& a, int num_sms, int smem_optin,
                               cudaStream_t stream);

// Dynamic shared memory that makes a CTA the only one resident on its SM
// (more than half of an SM's shared memory), so a grid of n CTAs occupies
// exactly n SMs.
constexpr size_t kExclusiveSmem = 120 * 1024;

}  // namespace ep
