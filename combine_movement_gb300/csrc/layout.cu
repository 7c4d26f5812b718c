// layout.cu -- per-expert histogram, exclusive prefix and stable per-(t,k)
// destination slot.
//
// DeepEP's dispatch call takes topk_idx and num_experts ("How DeepEP Utilizes
// TMA Instructions for Minimal SM Usage on Hopper GPUs", Practical Code
// Examples) and fills one contiguous receive buffer per expert. The pages do
// not show how the receive positions are computed; this library places the
// rows of expert e at offsets[e] .. offsets[e+1]-1 in ascending (t, k) order,
// which makes the result unique and the dispatch bit-reproducible.
//
// Entries are the T*K routing-table cells in row-major order (i = t*K + k).
// Large tables are cut into tiles of `warps * 32 * rounds` entries:
//   1. count  (one block per tile): shared-memory histogram -> tile_counts[e][tile]
//   2. scan   (one block): exclusive scan over the expert-major tile_counts,
//             giving each (expert, tile) its first receive row, plus counts
//             and offsets
//   3. rank   (one block per tile): each warp owns a contiguous run of the
//             tile; per-warp expert counts (warp match), a scan across warps,
//             then a second pass assigns ranks in entry order
// Tables of one tile take a single fused launch (count, scan and rank in one
// block). Only the histogram uses atomics, and counts do not depend on the
// order of the adds; every position is decided by scans, so the result is
// deterministic.
#include <cuda_runtime.h>

#include "../../include/ep.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace ep {
namespace {

constexpr unsigned kFullMask = 0xFFFFFFFFu;
constexpr size_t kRunSmemBudget = 64 * 1024;  // per-warp expert counters of the rank kernel
constexpr int kTileRounds = 4;                // rounds per warp per tile (multi-tile path)
constexpr int kFusedRounds = 8;               // rounds per warp for the single-block path
constexpr int kScanThreads = 1024;
constexpr int kCountThreads = 256;

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Expert id of a table cell, or -1 when the cell is masked (-1) or invalid.
__device__ __forceinline__ int expert_key(int64_t v, int E) {
    return (v >= 0 && v < E) ? static_cast<int>(v) : -1;
}

// Exclusive scan of one value per thread across the block (blockDim.x a
// multiple of 32, at most 1024). Returns the exclusive prefix; *total gets
// the block sum. Contains __syncthreads(); every thread must call it.
__device__ int64_t block_exclusive_scan(int64_t v, int64_t* total) {
    __shared__ int64_t warp_base[32];
    __shared__ int64_t block_total;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int64_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t o = __shfl_up_sync(kFullMask, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) warp_base[warp] = incl;  // warp sum
    __syncthreads();
    if (warp == 0) {
        const int64_t s = lane < nwarps ? warp_base[lane] : 0;
        int64_t si = s;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t o = __shfl_up_sync(kFullMask, si, d);
            if (lane >= d) si += o;
        }
        if (lane < nwarps) warp_base[lane] = si - s;  // exclusive warp base
        if (lane == 31) block_total = si;
    }
    __syncthreads();
    const int64_t out = warp_base[warp] + incl - v;
    *total = block_total;
    __syncthreads();  // the shared words may be reused by a later call
    return out;
}

// ---- 1. per-tile histogram -------------------------------------------------
__global__ void __launch_bounds__(kCountThreads) layout_count_kernel(
    const int64_t* __restrict__ idx, int64_t N, int E, int64_t tile, int num_tiles,
    int32_t* __restrict__ tile_counts, int32_t* status) {
    extern __shared__ int32_t hist[];
    for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t begin = tile * blockIdx.x;
    const int64_t end = min(N, begin + tile);
    bool bad = false;
    for (int64_t i = begin + threadIdx.x; i < end; i += blockDim.x) {
        const int64_t v = __ldg(idx + i);
        const int e = expert_key(v, E);
        if (e >= 0)
            atomicAdd(&hist[e], 1);
        else if (v != -1)
            bad = true;
    }
    if (bad) set_status(status, EP_ERR_BAD_EXPERT);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        tile_counts[static_cast<int64_t>(e) * num_tiles + blockIdx.x] = hist[e];
}

// ---- 2. scan over (expert, tile) --------------------------------------------
// In place: tile_counts[e][b] becomes the first receive row of expert e's
// entries in tile b.
__global__ void __launch_bounds__(kScanThreads) layout_scan_kernel(
    int32_t* __restrict__ tile_counts, int num_tiles, int E, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets) {
    const int64_t M = static_cast<int64_t>(E) * num_tiles;
    const int64_t per = (M + blockDim.x - 1) / blockDim.x;
    const int64_t lo = min(M, per * threadIdx.x), hi = min(M, lo + per);
    int64_t local = 0;
    for (int64_t i = lo; i < hi; ++i) local += tile_counts[i];
    int64_t total;
    int64_t run = block_exclusive_scan(local, &total);
    for (int64_t i = lo; i < hi; ++i) {
        const int32_t c = tile_counts[i];
        tile_counts[i] = static_cast<int32_t>(run);
        run += c;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t first = tile_counts[static_cast<int64_t>(e) * num_tiles];
        const int32_t next = (e + 1 < E) ? tile_counts[static_cast<int64_t>(e + 1) * num_tiles]
                                         : static_cast<int32_t>(total);
        offsets[e] = first;
        counts[e] = next - first;
    }
    if (threadIdx.x == 0) offsets[E] = static_cast<int32_t>(total);
}

// ---- 3. stable ranking (FUSED: also histogram + scan, single block) ----------
template <bool FUSED>
__global__ void layout_rank_kernel(const int64_t* __restrict__ idx, int64_t N, int E,
                                   int rounds, int64_t tile, int num_tiles,
                                   const int32_t* __restrict__ tile_base,
                                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                   int32_t* __restrict__ slot, int32_t* status) {
    extern __shared__ int32_t run[];  // [warps][E]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int64_t span = static_cast<int64_t>(rounds) * 32;
    const int64_t my_begin = tile * blockIdx.x + span * warp;
    int32_t* my = run + static_cast<int64_t>(warp) * E;

    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();

    // Pass A: per-warp expert counts over this warp's run of entries.
    bool bad = false;
    for (int r = 0; r < rounds; ++r) {
        const int64_t i = my_begin + static_cast<int64_t>(r) * 32 + lane;
        int key = -1;
        if (i < N) {
            const int64_t v = __ldg(idx + i);
            key = expert_key(v, E);
            if (key < 0 && v != -1) bad = true;
        }
        const uint32_t peers = __match_any_sync(kFullMask, key);
        if (key >= 0 && lane == __ffs(peers) - 1) my[key] += __popc(peers);
        __syncwarp();
    }
    if (FUSED && bad) set_status(status, EP_ERR_BAD_EXPERT);
    __syncthreads();

    if (FUSED) {
        // totals per expert, exclusive scan across experts, per-warp bases
        const int per = (E + blockDim.x - 1) / blockDim.x;
        const int e0 = min(E, per * static_cast<int>(threadIdx.x)), e1 = min(E, e0 + per);
        int64_t local = 0;
        for (int e = e0; e < e1; ++e)
            for (int w = 0; w < nwarps; ++w) local += run[static_cast<int64_t>(w) * E + e];
        int64_t total;
        int64_t base = block_exclusive_scan(local, &total);
        for (int e = e0; e < e1; ++e) {
            int64_t acc = base;
            for (int w = 0; w < nwarps; ++w) {
                const int32_t c = run[static_cast<int64_t>(w) * E + e];
                run[static_cast<int64_t>(w) * E + e] = static_cast<int32_t>(acc);
                acc += c;
            }
            offsets[e] = static_cast<int32_t>(base);
            counts[e] = static_cast<int32_t>(acc - base);
            base = acc;
        }
        if (threadIdx.x == 0) offsets[E] = static_cast<int32_t>(total);
    } else {
        for (int e = threadIdx.x; e < E; e += blockDim.x) {
            int32_t acc = tile_base[static_cast<int64_t>(e) * num_tiles + blockIdx.x];
            for (int w = 0; w < nwarps; ++w) {
                const int32_t c = run[static_cast<int64_t>(w) * E + e];
                run[static_cast<int64_t>(w) * E + e] = acc;
                acc += c;
            }
        }
    }
    __syncthreads();

    // Pass B: ranks in entry order. Within a round, lanes holding the same
    // expert are ordered by lane (= entry order); rounds run in order.
    for (int r = 0; r < rounds; ++r) {
        const int64_t i = my_begin + static_cast<int64_t>(r) * 32 + lane;
        int key = -1;
        if (i < N) key = expert_key(__ldg(idx + i), E);
        const uint32_t peers = __match_any_sync(kFullMask, key);
        if (i < N) slot[i] = key >= 0 ? my[key] + __popc(peers & lanemask_lt()) : -1;
        __syncwarp();
        if (key >= 0 && lane == __ffs(peers) - 1) my[key] += __popc(peers);
        __syncwarp();
    }
}

}  // namespace

LayoutPlan plan_layout(int64_t N, int E) {
    LayoutPlan p{};
    int warps = static_cast<int>(kRunSmemBudget / (sizeof(int32_t) * static_cast<size_t>(E)));
    warps = warps < 1 ? 1 : (warps > 32 ? 32 : warps);
    p.warps = warps;
    const int64_t fused_cap = static_cast<int64_t>(warps) * 32 * kFusedRounds;
    if (N <= fused_cap) {
        p.num_tiles = 1;
        p.rounds = static_cast<int>((N + 32LL * warps - 1) / (32LL * warps));
        if (p.rounds < 1) p.rounds = 1;
        p.tile = static_cast<int64_t>(warps) * 32 * p.rounds;
        p.workspace_bytes = 0;
    } else {
        p.rounds = kTileRounds;
        p.tile = static_cast<int64_t>(warps) * 32 * kTileRounds;
        p.num_tiles = static_cast<int>((N + p.tile - 1) / p.tile);
        p.workspace_bytes = sizeof(int32_t) * static_cast<size_t>(E) * p.num_tiles;
    }
    p.smem = sizeof(int32_t) * static_cast<size_t>(E) * warps;
    return p;
}

cudaError_t launch_layout(const int64_t* idx, int64_t N, int E, int32_t* counts,
                          int32_t* offsets, int32_t* slot, int32_t* tile_counts,
                          const LayoutPlan& p, int32_t* status, cudaStream_t stream) {
    const int threads = p.warps * 32;
    // The ranking kernel's dynamic shared memory can exceed the default 48 KB
    // (it also holds a few static words for the block scan).
    cudaError_t err = cudaFuncSetAttribute(p.num_tiles == 1 ? layout_rank_kernel<true>
                                                            : layout_rank_kernel<false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kRunSmemBudget));
    if (err != cudaSuccess) return err;
    if (p.num_tiles == 1) {
        layout_rank_kernel<true><<<1, threads, p.smem, stream>>>(
            idx, N, E, p.rounds, p.tile, 1, nullptr, counts, offsets, slot, status);
        return cudaGetLastError();
    }
    layout_count_kernel<<<p.num_tiles, kCountThreads, sizeof(int32_t) * E, stream>>>(
        idx, N, E, p.tile, p.num_tiles, tile_counts, status);
    layout_scan_kernel<<<1, kScanThreads, 0, stream>>>(tile_counts, p.num_tiles, E, counts,
                                                       offsets);
    layout_rank_kernel<false><<<p.num_tiles, threads, p.smem, stream>>>(
        idx, N, E, p.rounds, p.tile, p.num_tiles, tile_counts, counts, offsets, slot, status);
    return cudaGetLastError();
}

}  // namespace ep
