// combine_tma.cu -- combine with the K expert rows staged through a per-warp
// shared-memory ring by 1-D bulk copies (TMA), then reduced from shared
// memory.
//
// This applies the dispatch pattern of "How DeepEP Utilizes TMA Instructions
// for Minimal SM Usage on Hopper GPUs" (one elected lane issues bulk copies
// into its warp's private slice, completion on an mbarrier; sections
// "Per-Warp TMA Buffer Layout" and "Asynchronous Copy Primitives") to the
// other half of the MoE exchange. The copy engine keeps many kilobytes of
// expert rows in flight per warp without spending registers on them, which
// is what a small SM budget needs to cover memory latency. The ring is the
// two-stage overlap of the "tensor-memory-accelerator" atlas page ("Science
// and assumptions"): the loads of the next units proceed while the warp
// reduces the current one.
//
// Arithmetic is identical to the direct combine: fp32 accumulator from +0.0f,
// one fma per k in ascending k (skipped rows skipped), one bf16 RNE rounding.
//
// A unit is one C-byte column chunk of one token (C = kChunk, a multiple of
// 512). For unit j the elected lane bulk-loads the chunk of each of the
// token's K expert rows into stage j % NS (expect-tx = valid rows * bytes);
// all lanes wait on that stage's mbarrier, each lane reduces 16-byte columns
// from shared memory and writes them to y (a warp writes 512 contiguous
// bytes per step). Loads run NS-1 units ahead.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/ep.h"
#include "combine_math.cuh"
#include "kernels.cuh"
#include "ptx.cuh"

namespace ep {
namespace {

#ifndef EP_CTMA_STAGES
#define EP_CTMA_STAGES 4
#endif
#ifndef EP_CTMA_CHUNK
#define EP_CTMA_CHUNK 1024
#endif
#ifndef EP_CTMA_MAX_WARPS
#define EP_CTMA_MAX_WARPS 16
#endif

constexpr unsigned kFullMask = 0xFFFFFFFFu;
constexpr int kStages = EP_CTMA_STAGES;
constexpr uint32_t kChunk = EP_CTMA_CHUNK;
constexpr int kMaxWarps = EP_CTMA_MAX_WARPS;
constexpr uint32_t kColBytes = 512;
static_assert(kChunk % kColBytes == 0, "chunk must be whole 512-byte column blocks");

__host__ __device__ constexpr uint32_t barrier_region(int warps) {
    return (8u * kStages * warps + 127u) & ~127u;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

template <int KT>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) combine_tma_kernel(const CombineArgs a) {
    constexpr int NS = kStages;
    constexpr int P = NS - 1;
    constexpr uint32_t kStageBytes = KT * kChunk;
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const uint32_t bar0 = smem_u32(smem) + 8u * NS * warp;
    const uint32_t buf0 = smem_u32(smem) + barrier_region(nwarps) + kStageBytes * NS * warp;

    const bool leader = elect_one();
    const int leader_lane = __ffs(__ballot_sync(kFullMask, leader)) - 1;
    if (leader) {
#pragma unroll
        for (int s = 0; s < NS; ++s) mbar_init(bar0 + 8u * s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    griddep_wait();
    griddep_launch_dependents();

    const int64_t n_c = (a.row_bytes + kChunk - 1) / kChunk;
    const int64_t units = a.T * n_c;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * nwarps + warp;
    const int64_t nw_total = static_cast<int64_t>(gridDim.x) * nwarps;
    const int64_t u0 = units * gw / nw_total;
    const int64_t n = units * (gw + 1) / nw_total - u0;
    if (n <= 0) return;
    const uint64_t pol = policy_evict_first();

    // Lanes k < KT hold slot[t][k] (issue side, a token ahead too) and
    // slot/weight of the token being reduced (consume side).
    auto load_slot = [&](int64_t t) -> int32_t {
        if (t >= a.T || lane >= KT) return -1;
        int32_t s = __ldg(a.slot + t * KT + lane);
        if (s >= a.num_recv) {
            set_status(a.status, EP_ERR_BAD_SLOT);
            s = -1;
        }
        return s;
    };
    auto load_w = [&](int64_t t) -> float {
        return (t < a.T && lane < KT) ? __ldg(a.topk_w + t * KT + lane) : 0.0f;
    };

    int64_t i_tok = u0 / n_c;
    int32_t i_cur = load_slot(i_tok), i_next = load_slot(i_tok + 1);

    auto issue = [&](int64_t j) {
        const int64_t u = u0 + j;
        const int64_t t = u / n_c;
        if (t != i_tok) {
            i_tok = t;
            i_cur = i_next;
            i_next = load_slot(t + 1);
        }
        const uint32_t off = static_cast<uint32_t>(u - t * n_c) * kChunk;
        const uint32_t bytes = min(kChunk, a.row_bytes - off);
        const uint32_t valid = __ballot_sync(kFullMask, i_cur >= 0) & ((1u << KT) - 1u);
        const int s = static_cast<int>(j % NS);
        const uint32_t bar = bar0 + 8u * s;
        const uint32_t dst = buf0 + kStageBytes * s;
        if (leader) {
            fence_proxy_async_smem();  // the warp's reads of this stage precede the refill
            mbar_arrive_expect_tx(bar, __popc(valid) * bytes);
        }
#pragma unroll
        for (int k = 0; k < KT; ++k) {
            const int32_t sk = __shfl_sync(kFullMask, i_cur, k);
            if (leader && sk >= 0)
                bulk_load(dst + k * kChunk, a.expert_out + static_cast<int64_t>(sk) * a.row_bytes + off,
                          bytes, bar, pol);
        }
    };

    for (int64_t j = 0; j < P && j < n; ++j) issue(j);

    int64_t c_tok = u0 / n_c;
    int32_t c_s = load_slot(c_tok), c_s_next = load_slot(c_tok + 1);
    float c_w = load_w(c_tok), c_w_next = load_w(c_tok + 1);
    float wk[KT];
    bool on[KT];
#pragma unroll
    for (int k = 0; k < KT; ++k) {
        wk[k] = __shfl_sync(kFullMask, c_w, k);
        on[k] = __shfl_sync(kFullMask, c_s, k) >= 0;
    }

    for (int64_t j = 0; j < n; ++j) {
        if (j + P < n) issue(j + P);

        const int64_t u = u0 + j;
        const int64_t t = u / n_c;
        if (t != c_tok) {
            c_tok = t;
            c_s = c_s_next;
            c_w = c_w_next;
            c_s_next = load_slot(t + 1);
            c_w_next = load_w(t + 1);
#pragma unroll
            for (int k = 0; k < KT; ++k) {
                wk[k] = __shfl_sync(kFullMask, c_w, k);
                on[k] = __shfl_sync(kFullMask, c_s, k) >= 0;
            }
        }
        const int s = static_cast<int>(j % NS);
        uint32_t ok = 1;
        if (leader) ok = mbar_wait_bounded(bar0 + 8u * s, static_cast<uint32_t>((j / NS) & 1));
        ok = __shfl_sync(kFullMask, ok, leader_lane);
        if (!ok) {
            if (leader) {
                set_status(a.status, EP_ERR_TIMEOUT);
                mbar_drain_bounded<NS>(bar0, j, j + P < n ? j + P : n - 1);
            }
            break;
        }
        const uint32_t off = static_cast<uint32_t>(u - t * n_c) * kChunk;
        const uint32_t bytes = min(kChunk, a.row_bytes - off);
        const uint32_t src = buf0 + kStageBytes * s;
        uint8_t* yrow = a.y + t * static_cast<int64_t>(a.row_bytes) + off;
#pragma unroll
        for (uint32_t cb = 0; cb < kChunk; cb += kColBytes) {
            const uint32_t col = cb + lane * 16u;
            if (col < bytes) {
                float acc[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
                uint4 v[KT];
#pragma unroll
                for (int k = 0; k < KT; ++k) {
                    v[k] = make_uint4(0u, 0u, 0u, 0u);
                    if (on[k]) v[k] = lds128(src + k * kChunk + col);
                }
#pragma unroll
                for (int k = 0; k < KT; ++k)
                    if (on[k]) fma8(acc, wk[k], v[k]);
                st_v4(yrow + col, round8(acc));
            }
        }
        __syncwarp();
    }
}

template <int KT>
cudaError_t launch_kt(const CombineArgs& a, int num_sms, int smem_optin, cudaStream_t stream) {
    const size_t per_warp = static_cast<size_t>(KT) * kChunk * kStages;
    int warps = static_cast<int>((static_cast<size_t>(smem_optin) - barrier_region(kMaxWarps)) / per_warp);
    warps = warps > kMaxWarps ? kMaxWarps : warps;
    if (warps < 1) return cudaErrorInvalidConfiguration;
    size_t smem = barrier_region(warps) + per_warp * warps;
    if (smem < kExclusiveSmem) smem = kExclusiveSmem;
    auto kern = combine_tma_kernel<KT>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    const int64_t units = a.T * ((a.row_bytes + kChunk - 1) / kChunk);
    const int64_t ctas_needed = (units + warps - 1) / warps;
    const int grid = static_cast<int>(ctas_needed < num_sms ? ctas_needed : num_sms);
    if (grid <= 0) return cudaSuccess;
    return launch_dependent(kern, grid, warps * 32, smem, stream, a);
}

}  // namespace

bool combine_tma_supported(int K) { return K >= 1 && K <= 8; }

cudaError_t launch_combine_tma(const CombineArgs& a, int num_sms, int smem_optin,
                               cudaStream_t stream) {
    switch (a.K) {
        case 1: return launch_kt<1>(a, num_sms, smem_optin, stream);
        case 2: return launch_kt<2>(a, num_sms, smem_optin, stream);
        case 3: return launch_kt<3>(a, num_sms, smem_optin, stream);
        case 4: return launch_kt<4>(a, num_sms, smem_optin, stream);
        case 5: return launch_kt<5>(a, num_sms, smem_optin, stream);
        case 6: return launch_kt<6>(a, num_sms, smem_optin, stream);
        case 7: return launch_kt<7>(a, num_sms, smem_optin, stream);
        case 8: return launch_kt<8>(a, num_sms, smem_optin, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ep
