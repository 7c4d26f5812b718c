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
// The table is cut into tiles of `warps * 32 * rounds` entries:
//   1. tile kernel (one block per tile): loads the tile's ids once, counts
//      them per warp (warp match), scans across warps and assigns every entry
//      its rank among the tile's entries of the same expert, in entry order;
//      writes the tile's per-expert counts to tile_counts[e][tile] and the
//      packed (rank, expert) into slot.
//   2. finish kernel (one block per tile): computes, from the small
//      [E][tiles] array, each expert's first row and the rows taken by
//      earlier tiles (every block does this itself, saving a launch), then
//      rewrites each packed entry as its final slot; block 0 writes counts
//      and offsets. Very large tables scan once in a separate one-block
//      kernel instead.
// A table that fits one tile takes a single fused launch. No position
// depends on the order of concurrent operations (there are no atomics; the
// per-warp counts are owned by their warp), so the result is deterministic.
#include <cuda_runtime.h>

#include "../../include/ep.h"
#include "kernels.cuh"
#include "ptx.cuh"

namespace ep {
namespace {

constexpr unsigned kFullMask = 0xFFFFFFFFu;
constexpr size_t kRunSmemBudget = 64 * 1024;  // per-warp expert counters of the tile kernel
constexpr int kMaxRounds = 8;                 // 32-entry rounds per warp per tile, at most
constexpr int kTargetTiles = 128;             // tiles to aim for before rounds grow
constexpr int kMaxRedundantTiles = 512;       // above this, one block scans for everyone
constexpr int kScanThreads = 1024;
constexpr int kFinishThreads = 512;
constexpr int kExpertBits = 12;               // packed entry: (rank << 12) | expert, E <= 4096
constexpr int32_t kExpertMask = (1 << kExpertBits) - 1;
static_assert((1 << kExpertBits) >= EP_MAX_EXPERTS, "expert id must fit the packed entry");

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

// ---- tile kernel: per-warp counts, per-tile ranks ----------------------------
// Every warp owns `rounds` consecutive 32-entry rounds of its tile; all of
// its routing ids are loaded up front (one memory latency, not one per
// round). Pass A counts ids per warp (warp match: one shared-memory add per
// distinct id per round); a scan across the warps turns the counts into
// per-warp starting ranks; pass B hands out ranks in entry order.
//  FUSED (the whole table is one tile): the block also scans across experts
//    and writes counts, offsets and final slots.
//  otherwise: writes the tile's per-expert counts to tile_counts[e][tile]
//    and, per entry, (rank within the tile << 12) | expert into slot, which
//    layout_finish_kernel turns into the final slot.
template <bool FUSED>
__global__ void layout_tile_kernel(const int64_t* __restrict__ idx, int64_t N, int E, int rounds,
                                   int num_tiles, int32_t* __restrict__ tile_counts,
                                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                   int32_t* __restrict__ slot, int32_t* status) {
    extern __shared__ int32_t run[];  // [warps][E]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int64_t tile = static_cast<int64_t>(nwarps) * 32 * rounds;
    const int64_t wbase = tile * blockIdx.x + static_cast<int64_t>(warp) * 32 * rounds;

    int key[kMaxRounds];
    bool bad = false;
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        key[r] = -1;
        const int64_t i = wbase + r * 32 + lane;
        if (r < rounds && i < N) {
            const int64_t v = __ldg(idx + i);
            key[r] = expert_key(v, E);
            bad |= (key[r] < 0 && v != -1);
        }
    }
    int32_t* my = run + static_cast<int64_t>(warp) * E;
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        if (r < rounds) {
            const uint32_t peers = __match_any_sync(kFullMask, key[r]);
            if (key[r] >= 0 && lane == __ffs(peers) - 1) my[key[r]] += __popc(peers);
            __syncwarp();
        }
    }
    if (bad) set_status(status, EP_ERR_BAD_EXPERT);
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
            int32_t acc = 0;
            for (int w = 0; w < nwarps; ++w) {
                const int32_t c = run[static_cast<int64_t>(w) * E + e];
                run[static_cast<int64_t>(w) * E + e] = acc;
                acc += c;
            }
            tile_counts[static_cast<int64_t>(e) * num_tiles + blockIdx.x] = acc;
        }
    }
    __syncthreads();

#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        if (r < rounds) {
            const int64_t i = wbase + r * 32 + lane;
            const int k = key[r];
            const uint32_t peers = __match_any_sync(kFullMask, k);
            if (i < N) {
                if (k >= 0) {
                    const int32_t rank = my[k] + __popc(peers & lanemask_lt());
                    slot[i] = FUSED ? rank : ((rank << kExpertBits) | k);
                } else {
                    slot[i] = -1;
                }
            }
            __syncwarp();
            if (k >= 0 && lane == __ffs(peers) - 1) my[k] += __popc(peers);
            __syncwarp();
        }
    }
}

// ---- scan over (expert, tile), one block (large tables only) -----------------
// In place: tile_counts[e][b] becomes the first receive row of expert e's
// entries in tile b; also writes counts and offsets.
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

// ---- finish kernel: final slots ------------------------------------------------
// One block per tile. Unless PRESCANNED, every block computes the prefix it
// needs itself (expert totals and the counts of earlier tiles, read from the
// small [E][tiles] array; one scan across experts), which saves a launch;
// block 0 also writes counts and offsets. Then each packed entry becomes
// base[expert] + rank.
template <bool PRESCANNED>
__global__ void __launch_bounds__(kFinishThreads) layout_finish_kernel(
    const int32_t* __restrict__ tile_counts, int num_tiles, int E, int64_t N, int64_t tile,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ slot) {
    extern __shared__ int32_t base[];  // [E] (+ [E] of totals when !PRESCANNED)
    if (PRESCANNED) {
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            base[e] = tile_counts[static_cast<int64_t>(e) * num_tiles + blockIdx.x];
    } else {
        int32_t* tot = base + E;
        const int per = (E + blockDim.x - 1) / blockDim.x;
        const int e0 = min(E, per * static_cast<int>(threadIdx.x)), e1 = min(E, e0 + per);
        int64_t local = 0;
        for (int e = e0; e < e1; ++e) {
            const int32_t* row = tile_counts + static_cast<int64_t>(e) * num_tiles;
            int32_t t = 0, before = 0;
            for (int b = 0; b < num_tiles; ++b) {
                const int32_t c = __ldg(row + b);
                t += c;
                before += b < static_cast<int>(blockIdx.x) ? c : 0;
            }
            tot[e] = t;
            base[e] = before;
            local += t;
        }
        int64_t total;
        int64_t off = block_exclusive_scan(local, &total);
        for (int e = e0; e < e1; ++e) {
            if (blockIdx.x == 0) {
                offsets[e] = static_cast<int32_t>(off);
                counts[e] = tot[e];
            }
            base[e] += static_cast<int32_t>(off);
            off += tot[e];
        }
        if (blockIdx.x == 0 && threadIdx.x == 0) offsets[E] = static_cast<int32_t>(total);
    }
    __syncthreads();
    const int64_t begin = tile * blockIdx.x;
    const int64_t end = min(N, begin + tile);
    for (int64_t i = begin + threadIdx.x; i < end; i += blockDim.x) {
        const int32_t p = slot[i];
        if (p >= 0) slot[i] = base[p & kExpertMask] + (p >> kExpertBits);
    }
}

}  // namespace

LayoutPlan plan_layout(int64_t N, int E) {
    LayoutPlan p{};
    int warps = static_cast<int>(kRunSmemBudget / (sizeof(int32_t) * static_cast<size_t>(E)));
    warps = warps < 1 ? 1 : (warps > 32 ? 32 : warps);
    p.warps = warps;
    const int64_t per_round = 32LL * warps;  // entries per round of the whole block
    if (N <= per_round * kMaxRounds) {
        p.num_tiles = 1;
        p.rounds = static_cast<int>((N + per_round - 1) / per_round);
        if (p.rounds < 1) p.rounds = 1;
    } else {
        int64_t r = (N + per_round * kTargetTiles - 1) / (per_round * kTargetTiles);
        p.rounds = static_cast<int>(r < 1 ? 1 : (r > kMaxRounds ? kMaxRounds : r));
    }
    p.tile = per_round * p.rounds;
    if (N > per_round * kMaxRounds) p.num_tiles = static_cast<int>((N + p.tile - 1) / p.tile);
    p.workspace_bytes =
        p.num_tiles > 1 ? sizeof(int32_t) * static_cast<size_t>(E) * p.num_tiles : 0;
    p.smem = sizeof(int32_t) * static_cast<size_t>(E) * warps;
    return p;
}

cudaError_t launch_layout(const int64_t* idx, int64_t N, int E, int32_t* counts,
                          int32_t* offsets, int32_t* slot, int32_t* tile_counts,
                          const LayoutPlan& p, int32_t* status, cudaStream_t stream) {
    const int threads = p.warps * 32;
    // The tile kernel's dynamic shared memory can exceed the default 48 KB
    // (it also holds a few static words for the block scan).
    cudaError_t err = cudaFuncSetAttribute(
        p.num_tiles == 1 ? layout_tile_kernel<true> : layout_tile_kernel<false>,
        cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kRunSmemBudget));
    if (err != cudaSuccess) return err;
    if (p.num_tiles == 1) {
        layout_tile_kernel<true><<<1, threads, p.smem, stream>>>(idx, N, E, p.rounds, 1, nullptr,
                                                                 counts, offsets, slot, status);
        return cudaGetLastError();
    }
    layout_tile_kernel<false><<<p.num_tiles, threads, p.smem, stream>>>(
        idx, N, E, p.rounds, p.num_tiles, tile_counts, counts, offsets, slot, status);
    if (p.num_tiles <= kMaxRedundantTiles) {
        layout_finish_kernel<false><<<p.num_tiles, kFinishThreads, 2 * sizeof(int32_t) * E, stream>>>(
            tile_counts, p.num_tiles, E, N, p.tile, counts, offsets, slot);
    } else {
        layout_scan_kernel<<<1, kScanThreads, 0, stream>>>(tile_counts, p.num_tiles, E, counts,
                                                           offsets);
        layout_finish_kernel<true><<<p.num_tiles, kFinishThreads, sizeof(int32_t) * E, stream>>>(
            tile_counts, p.num_tiles, E, N, p.tile, counts, offsets, slot);
    }
    return cudaGetLastError();
}

}  // namespace ep
