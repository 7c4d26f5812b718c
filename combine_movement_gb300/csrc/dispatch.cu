// dispatch.cu -- copy every token row into the receive row of each of its
// top-k experts with 1-D bulk copies (TMA) through a per-warp shared-memory
// ring.
//
// Pattern ("How DeepEP Utilizes TMA Instructions for Minimal SM Usage on
// Hopper GPUs"): each warp owns a private slice of dynamic shared memory
// ("Per-Warp TMA Buffer Layout"); one elected lane bulk-loads a row chunk
// into it, completion is tracked on an mbarrier, and the same lane
// bulk-stores it back out, waiting on the bulk group before the slice is
// reused ("Asynchronous Copy Primitives"). The kernel asks for its shared
// memory through the max-dynamic-shared-memory attribute, sized from the
// per-warp slice ("Dynamic Shared Memory Configuration").
//
// What differs from the page's receive loop, and why:
//  * Each chunk is loaded ONCE and stored K times (one store per expert that
//    receives the token); the page's loop moves one received copy per
//    load, which on one GPU would read x K times.
//  * The slice is a ring of NS stages with P loads kept in flight ahead of
//    the stores (the two-stage overlap of the "tensor-memory-accelerator"
//    atlas page, "Science and assumptions"), instead of a load / wait / store
//    sequence per half row.
//  * Rows are cut into equal 16-byte-multiple chunks that fit a stage rather
//    than fixed halves, so any hidden size with H % 8 == 0 works.
//  * Work is split as contiguous, equal ranges of (token, chunk) units per
//    warp over a persistent grid of one CTA per SM (the SM budget).
#include <cuda_runtime.h>

#include "../../include/ep.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace ep {
namespace {

// Build-time shape of the ring (defaults are the tuned values).
#ifndef EP_DISPATCH_WARPS
#define EP_DISPATCH_WARPS 8
#endif
#ifndef EP_DISPATCH_STAGES
#define EP_DISPATCH_STAGES 4
#endif
#ifndef EP_DISPATCH_PREFETCH
#define EP_DISPATCH_PREFETCH 2
#endif

constexpr unsigned kFullMask = 0xFFFFFFFFu;
constexpr int kDispatchWarps = EP_DISPATCH_WARPS;

// Bytes reserved in front of the stages for the mbarriers (8 B per stage per
// warp), rounded up so every stage starts 128-byte aligned.
__host__ __device__ constexpr uint32_t barrier_region(int stages, int warps) {
    return (8u * stages * warps + 127u) & ~127u;
}

template <int NS, int P>
__global__ void __launch_bounds__(kDispatchWarps * 32, 1) dispatch_kernel(const DispatchArgs a) {
    static_assert(P >= 1 && P < NS, "need 1 <= P < NS");
    extern __shared__ __align__(128) uint8_t smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;

    const uint32_t bar0 = smem_u32(smem) + 8u * NS * warp;
    const uint32_t buf0 = smem_u32(smem) + barrier_region(NS, nwarps) +
                          static_cast<uint32_t>(NS) * a.stage_bytes * warp;

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

    const int64_t units = a.T * static_cast<int64_t>(a.n_chunks);
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * nwarps + warp;
    const int64_t nw_total = static_cast<int64_t>(gridDim.x) * nwarps;
    const int64_t u0 = units * gw / nw_total;
    const int64_t n = units * (gw + 1) / nw_total - u0;
    if (n <= 0) return;

    const uint64_t pol_load = policy_evict_first();
    const uint64_t pol_store = policy_evict_normal();

    // Bulk-load local unit j (token, chunk) into its ring stage.
    auto issue_load = [&](int64_t j) {
        if (!leader) return;
        const int64_t u = u0 + j;
        const int64_t t = u / a.n_chunks;
        const uint32_t off = static_cast<uint32_t>(u - t * a.n_chunks) * a.chunk_bytes;
        const uint32_t bytes = min(a.chunk_bytes, a.row_bytes - off);
        const int s = static_cast<int>(j % NS);
        const uint32_t bar = bar0 + 8u * s;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(buf0 + static_cast<uint32_t>(s) * a.stage_bytes,
                  a.x + t * static_cast<int64_t>(a.row_bytes) + off, bytes, bar, pol_load);
    };

    // Lanes k < K hold slot[t][k] (and topk_w[t][k]) of the current token and
    // of the next one, loaded a token ahead.
    auto load_slot = [&](int64_t t) -> int32_t {
        return (t < a.T && lane < a.K) ? __ldg(a.slot + t * a.K + lane) : -1;
    };
    auto load_w = [&](int64_t t) -> float {
        return (a.topk_w != nullptr && t < a.T && lane < a.K) ? __ldg(a.topk_w + t * a.K + lane)
                                                              : 0.0f;
    };

    for (int64_t j = 0; j < P && j < n; ++j) issue_load(j);

    int64_t tok = u0 / a.n_chunks;
    int32_t s_cur = load_slot(tok), s_next = load_slot(tok + 1);
    float w_cur = load_w(tok), w_next = load_w(tok + 1);

    for (int64_t j = 0; j < n; ++j) {
        const int64_t u = u0 + j;
        const int64_t t = u / a.n_chunks;
        const uint32_t c = static_cast<uint32_t>(u - t * a.n_chunks);
        if (t != tok) {
            tok = t;
            s_cur = s_next;
            w_cur = w_next;
            s_next = load_slot(t + 1);
            w_next = load_w(t + 1);
        }

        // Refill: the stage of unit j+P was last used by unit j+P-NS; its
        // stores must have finished reading shared memory.
        if (j + P < n) {
            if (leader) bulk_wait_read<NS - P - 1>();
            issue_load(j + P);
        }

        const int s = static_cast<int>(j % NS);
        uint32_t ok = 1;
        if (leader) ok = mbar_wait_bounded(bar0 + 8u * s, static_cast<uint32_t>((j / NS) & 1));
        ok = __shfl_sync(kFullMask, ok, leader_lane);
        if (!ok) {
            if (leader) set_status(a.status, EP_ERR_TIMEOUT);
            break;
        }

        const uint32_t off = c * a.chunk_bytes;
        const uint32_t bytes = min(a.chunk_bytes, a.row_bytes - off);
        const uint32_t src = buf0 + static_cast<uint32_t>(s) * a.stage_bytes;
        for (int k = 0; k < a.K; ++k) {
            const int32_t d = __shfl_sync(kFullMask, s_cur, k);
            if (leader && d >= 0) {
                if (d < a.num_recv)
                    bulk_store(a.recv_x + static_cast<int64_t>(d) * a.row_bytes + off, src, bytes,
                               pol_store);
                else
                    set_status(a.status, EP_ERR_BAD_SLOT);
            }
        }
        if (leader) bulk_commit();

        // Routing metadata of each received row, once per (t, k).
        if (c == 0 && lane < a.K && s_cur >= 0 && s_cur < a.num_recv) {
            if (a.recv_w != nullptr) a.recv_w[s_cur] = w_cur;
            if (a.recv_src != nullptr) a.recv_src[s_cur] = static_cast<int32_t>(t * a.K + lane);
        }
    }
    // Shared memory must outlive every bulk store that reads it.
    if (leader) bulk_wait<0>();
}

// ---- ablation: the same copy through the load/store units ---------------------
// Every lane moves 16-byte vectors with plain ld.global / st.global: a warp
// loads kLsuBlocks 512-byte column blocks of a row into registers and stores
// them to each of the K receive rows. This is the register-staged copy the
// pages contrast TMA with ("How DeepEP Utilizes TMA Instructions for Minimal
// SM Usage on Hopper GPUs", Summary and FAQ: the UNROLLED_WARP_COPY path of
// pre-Hopper GPUs; TMA study note, history of copying). Built only with
// EP_DISPATCH_MODE=1, for measuring what the bulk-copy path saves; it moves
// the rows only (no recv_w / recv_src).
#ifndef EP_DISPATCH_MODE
#define EP_DISPATCH_MODE 0
#endif
#ifndef EP_LSU_THREADS
#define EP_LSU_THREADS 512
#endif
#ifndef EP_LSU_BLOCKS
#define EP_LSU_BLOCKS 4
#endif
constexpr int kLsuThreads = EP_LSU_THREADS;
constexpr int kLsuBlocks = EP_LSU_BLOCKS;

__global__ void __launch_bounds__(kLsuThreads, 1) dispatch_lsu_kernel(const DispatchArgs a) {
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    constexpr uint32_t kUnit = 512u * kLsuBlocks;
    const int64_t n_cb = (a.row_bytes + kUnit - 1) / kUnit;
    const int64_t units = a.T * n_cb;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * nwarps + warp;
    const int64_t nw_total = static_cast<int64_t>(gridDim.x) * nwarps;
    const int64_t u0 = units * gw / nw_total, u1 = units * (gw + 1) / nw_total;
    int64_t tok = -1;
    int32_t s_lane = -1;
    for (int64_t u = u0; u < u1; ++u) {
        const int64_t t = u / n_cb;
        const uint32_t col0 = static_cast<uint32_t>(u - t * n_cb) * kUnit + lane * 16u;
        if (t != tok) {
            tok = t;
            s_lane = lane < a.K ? __ldg(a.slot + t * a.K + lane) : -1;
        }
        uint4 v[kLsuBlocks];
        const uint8_t* src = a.x + t * static_cast<int64_t>(a.row_bytes);
#pragma unroll
        for (int b = 0; b < kLsuBlocks; ++b) {
            v[b] = make_uint4(0u, 0u, 0u, 0u);
            if (col0 + b * 512u < a.row_bytes) v[b] = ld_nc_v4(src + col0 + b * 512u);
        }
        for (int k = 0; k < a.K; ++k) {
            const int32_t d = __shfl_sync(kFullMask, s_lane, k);
            if (d < 0) continue;
            if (d >= a.num_recv) {
                if (lane == 0) set_status(a.status, EP_ERR_BAD_SLOT);
                continue;
            }
            uint8_t* dst = a.recv_x + static_cast<int64_t>(d) * a.row_bytes;
#pragma unroll
            for (int b = 0; b < kLsuBlocks; ++b)
                if (col0 + b * 512u < a.row_bytes) st_v4(dst + col0 + b * 512u, v[b]);
        }
    }
}

// Ring shape compiled in: stages per warp, loads in flight ahead.
constexpr int kStages = EP_DISPATCH_STAGES;
constexpr int kPrefetch = EP_DISPATCH_PREFETCH;

}  // namespace

cudaError_t launch_dispatch(const DispatchArgs& a, int num_sms, int smem_optin,
                            cudaStream_t stream) {
    (void)smem_optin;
    if (EP_DISPATCH_MODE == 1) {
        cudaError_t e = cudaFuncSetAttribute(dispatch_lsu_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(kExclusiveSmem));
        if (e != cudaSuccess) return e;
        return launch_dependent(dispatch_lsu_kernel, num_sms, kLsuThreads, kExclusiveSmem, stream, a);
    }
    const size_t smem = static_cast<size_t>(barrier_region(kStages, kDispatchWarps)) +
                        static_cast<size_t>(kDispatchWarps) * kStages * a.stage_bytes;
    const size_t request = smem < kExclusiveSmem ? kExclusiveSmem : smem;
    auto kern = dispatch_kernel<kStages, kPrefetch>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(request));
    if (err != cudaSuccess) return err;
    const int64_t units = a.T * static_cast<int64_t>(a.n_chunks);
    int64_t ctas_needed = (units + kDispatchWarps - 1) / kDispatchWarps;
    const int grid = static_cast<int>(ctas_needed < num_sms ? ctas_needed : num_sms);
    if (grid <= 0) return cudaSuccess;
    return launch_dependent(kern, grid, kDispatchWarps * 32, request, stream, a);
}

// Stage size the host plans rows with: the per-warp slice split into the
// ring's stages, rounded down to 16 bytes.
uint32_t dispatch_stage_capacity(int smem_optin) {
    const size_t per_warp =
        (static_cast<size_t>(smem_optin) - barrier_region(kStages, kDispatchWarps)) / kDispatchWarps;
    return static_cast<uint32_t>((per_warp / kStages) & ~static_cast<size_t>(15));
}

}  // namespace ep
