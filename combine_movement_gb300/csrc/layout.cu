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
//      them per warp (ballot peer groups), scans across warps and assigns every entry
//      its rank among the tile's entries of the same expert, in entry order;
//      writes the tile's per-expert counts to tile_counts[tile][e] and the
//      packed (rank, expert) into slot.
//   2. finish kernel (one block per tile): computes, from the small
//      [tiles][E] table, each expert's first row and the rows taken by
//      earlier tiles (every block does this itself, saving a launch), then
//      rewrites each packed entry as its final slot; block 0 writes counts
//      and offsets. Very large tables scan once in a separate one-block
//      kernel instead.
// A table that fits one tile takes a single fused launch. No position
// depends on the order of concurrent operations: per-warp counts are owned
// by their warp, and the only atomics are integer sums (order-free), so the
// result is deterministic.
#include <cuda_runtime.h>
#include <unistd.h>

#include <chrono>

#include "../../include/ep.h"
#include "kernels.cuh"
#include "ptx.cuh"
#include "routing.cuh"

namespace ep {
namespace {

constexpr size_t kRunSmemBudget = 64 * 1024;  // per-warp expert counters of the tile kernel
constexpr int kMaxRounds = 8;                 // 32-entry rounds per warp per tile, at most
constexpr int kFusedRounds = 1;               // one block alone up to this many rounds
#ifndef EP_LAYOUT_SINGLE_ROUNDS
#define EP_LAYOUT_SINGLE_ROUNDS 4
#endif
constexpr int kSingleRounds = EP_LAYOUT_SINGLE_ROUNDS;  // target rounds per warp then
static_assert(kSingleRounds >= 1 && kSingleRounds <= 8, "single-block rounds in [1, 8]");
constexpr int kTargetTiles = 128;             // tiles to aim for before rounds grow
constexpr int kMaxRedundantTiles = 512;       // above this, one block scans for everyone
constexpr int kCoopMaxTiles = 128;            // tables of at most this many tiles: one launch
constexpr int kScanThreads = 1024;
constexpr int kFinishThreads = 512;
constexpr int kExpertBits = 12;               // packed entry: (rank << 12) | expert, E <= 4096
constexpr int32_t kExpertMask = (1 << kExpertBits) - 1;
static_assert((1 << kExpertBits) >= EP_MAX_EXPERTS, "expert id must fit the packed entry");

// Exclusive scan across the block's warps of the per-warp counts
// run[w][e], one expert per thread (in place); writes the tile total of
// each expert to out[e * stride]. Loads are batched 8 warps at a
// time so the chain does not wait on shared memory once per warp.
__device__ __forceinline__ void scan_across_warps(int32_t* run, int E, int nwarps,
                                                  int32_t* out, int64_t stride) {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t acc = 0;
        for (int w0 = 0; w0 < nwarps; w0 += 8) {
            int32_t c[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                c[u] = w0 + u < nwarps ? run[static_cast<int64_t>(w0 + u) * E + e] : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (w0 + u < nwarps) {
                    run[static_cast<int64_t>(w0 + u) * E + e] = acc;
                    acc += c[u];
                }
            }
        }
        out[static_cast<int64_t>(e) * stride] = acc;
    }
}

// ---- tile kernel: per-warp counts, per-tile ranks ----------------------------
// Every warp owns `rounds` consecutive 32-entry rounds of its tile; all of
// its routing ids are loaded up front (one memory latency, not one per
// round). Pass A counts ids per warp (ballot peer groups: one shared-memory
// add per distinct id per round); a scan across the warps turns the counts into
// per-warp starting ranks; pass B hands out ranks in entry order.
//  FUSED (the whole table is one tile): the block also scans across experts
//    and writes counts, offsets and final slots.
//  otherwise: writes the tile's per-expert counts to tile_counts[tile][e]
//    and, per entry, (rank within the tile << 12) | expert into slot, which
//    layout_finish_kernel turns into the final slot.
template <bool FUSED>
__global__ void __launch_bounds__(1024) layout_tile_kernel(const int64_t* __restrict__ idx, int64_t N, int E, int rounds,
                                   int num_tiles, int32_t* __restrict__ tile_counts,
                                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                   int32_t* __restrict__ slot, int32_t* status) {
    extern __shared__ int32_t run[];  // [warps][E]
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int64_t tile = static_cast<int64_t>(nwarps) * 32 * rounds;
    const int64_t wbase = tile * blockIdx.x + static_cast<int64_t>(warp) * 32 * rounds;
    const int kbits = key_bits_for(E);

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
    // one pass: ranks within the warp and the warp's per-expert counts
    int32_t rank[kMaxRounds];
    int32_t* my = run + static_cast<int64_t>(warp) * E;
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        rank[r] = 0;
        if (r < rounds) {
            const int k = key[r];
            const uint32_t peers = peers_of(k, kbits);
            if (k >= 0) rank[r] = my[k] + __popc(peers & lanemask_lt());
            __syncwarp();
            if (k >= 0 && lane == __ffs(peers) - 1) my[k] += __popc(peers);
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
        scan_across_warps(run, E, nwarps, tile_counts + static_cast<int64_t>(blockIdx.x) * E, 1);
    }
    __syncthreads();

    // my[] now holds each warp's first rank per expert (plus the expert's
    // first row when FUSED)
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        const int64_t i = wbase + r * 32 + lane;
        if (r < rounds && i < N) {
            const int k = key[r];
            if (k >= 0) {
                const int32_t rk = my[k] + rank[r];
                slot[i] = FUSED ? rk : ((rk << kExpertBits) | k);
            } else {
                slot[i] = -1;
            }
        }
    }
}

// ---- scan over (expert, tile), one block (large tables only) -----------------
// In place over the tile-major table: tile_counts[b][e] becomes the first
// receive row of expert e's entries in tile b (experts in order, tiles in
// order within an expert); also writes counts and offsets.
__global__ void __launch_bounds__(kScanThreads) layout_scan_kernel(
    int32_t* __restrict__ tile_counts, int num_tiles, int E, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t M = static_cast<int64_t>(E) * num_tiles;
    const int64_t per = (M + blockDim.x - 1) / blockDim.x;
    const int64_t lo = min(M, per * threadIdx.x), hi = min(M, lo + per);
    // position q of the expert-major order lives at [q % tiles][q / tiles]
    auto at = [&](int64_t q) -> int32_t& {
        return tile_counts[(q % num_tiles) * E + q / num_tiles];
    };
    int64_t local = 0;
    for (int64_t q = lo; q < hi; ++q) local += at(q);
    int64_t total;
    int64_t run = block_exclusive_scan(local, &total);
    for (int64_t q = lo; q < hi; ++q) {
        const int32_t c = at(q);
        at(q) = static_cast<int32_t>(run);
        run += c;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t first = tile_counts[e];
        const int32_t next = (e + 1 < E) ? tile_counts[e + 1] : static_cast<int32_t>(total);
        offsets[e] = first;
        counts[e] = next - first;
    }
    if (threadIdx.x == 0) offsets[E] = static_cast<int32_t>(total);
}

// ---- finish kernel: final slots ------------------------------------------------
// One block per tile. Unless PRESCANNED, every block computes the prefix it
// needs itself (expert totals and the counts of earlier tiles, read from the
// small [tiles][E] table; one scan across experts), which saves a launch;
// block 0 also writes counts and offsets. Then each packed entry becomes
// base[expert] + rank.
template <bool PRESCANNED>
__global__ void __launch_bounds__(kFinishThreads) layout_finish_kernel(
    const int32_t* __restrict__ tile_counts, int num_tiles, int E, int64_t N, int64_t tile,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ slot) {
    extern __shared__ int32_t base[];  // [E] (+ [E] of totals when !PRESCANNED)
    griddep_wait();
    griddep_launch_dependents();
    if (PRESCANNED) {
        for (int e = threadIdx.x; e < E; e += blockDim.x)
            base[e] = tile_counts[static_cast<int64_t>(blockIdx.x) * E + e];
    } else {
        int32_t* tot = base + E;
        for (int e = threadIdx.x; e < E; e += blockDim.x) tot[e] = base[e] = 0;
        __syncthreads();
        // Expert totals and the rows taken by earlier tiles: one coalesced
        // pass over the [tiles][E] counts, loads batched ahead of the
        // (order-free) integer shared-memory adds.
        const int64_t M = static_cast<int64_t>(E) * num_tiles;
        constexpr int kBatch = 8;
        for (int64_t f0 = threadIdx.x; f0 < M; f0 += static_cast<int64_t>(blockDim.x) * kBatch) {
            int32_t c[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t f = f0 + static_cast<int64_t>(u) * blockDim.x;
                c[u] = f < M ? __ldg(tile_counts + f) : 0;
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t f = f0 + static_cast<int64_t>(u) * blockDim.x;
                if (f < M && c[u] != 0) {
                    const int b = static_cast<int>(f / E);
                    const int e = static_cast<int>(f - static_cast<int64_t>(b) * E);
                    atomicAdd(&tot[e], c[u]);
                    if (b < static_cast<int>(blockIdx.x)) atomicAdd(&base[e], c[u]);
                }
            }
        }
        __syncthreads();
        const int per = (E + blockDim.x - 1) / blockDim.x;
        const int e0 = min(E, per * static_cast<int>(threadIdx.x)), e1 = min(E, e0 + per);
        int64_t local = 0;
        for (int e = e0; e < e1; ++e) local += tot[e];
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

// ---- single-cluster layout ---------------------------------------------------
// For tables that fit kClusterCtas tiles (up to 8 rounds per warp), one
// thread-block cluster does the whole layout. Its CTAs are co-scheduled on
// one GPC, so the tiles' per-expert counts are exchanged through distributed
// shared memory and the hardware cluster barrier, with no global round trips
// and no workspace:
//   phase 1  as in the other kernels: ids, per-warp ranks and counts, tile
//            counts into this CTA's shared memory
//   barrier  (cluster)
//   phase 2  every CTA reads each CTA's tile counts (DSMEM): expert totals and
//            the rows of earlier tiles
//   barrier  (cluster; after it no CTA reads another's shared memory, so each
//            may finish and exit on its own)
//   phase 3  scan across experts, final slots; CTA 0 writes counts, offsets.
constexpr int kClusterCtas = 8;  // portable cluster size
// Non-portable cluster size for the wider variant (plan_layout_wide_cluster).
constexpr int kWideClusterCtas = 16;

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// shared::cluster address of `local` (this CTA's shared memory) in CTA `rank`
__device__ __forceinline__ uint32_t cluster_map(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ int32_t ld_cluster(uint32_t addr) {
    int32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

template <int CTAS>
__global__ void __launch_bounds__(1024) layout_cluster_kernel(
    const int64_t* __restrict__ idx, int64_t N, int E, int rounds, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ slot, int32_t* status) {
    extern __shared__ int32_t run[];  // [warps][E] per-warp counts, then [E] tile counts
    griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int tile_id = static_cast<int>(cluster_rank());
    const int ntiles = static_cast<int>(gridDim.x);  // the grid is one cluster
    const int64_t tile = static_cast<int64_t>(nwarps) * 32 * rounds;
    const int64_t wbase = tile * tile_id + static_cast<int64_t>(warp) * 32 * rounds;
    const int kbits = key_bits_for(E);
    int32_t* tile_tot = run + static_cast<int64_t>(nwarps) * E;

    int key[kMaxRounds];
    int32_t rank[kMaxRounds];
    bool bad = false;
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        key[r] = -1;
        rank[r] = 0;
        const int64_t i = wbase + r * 32 + lane;
        if (r < rounds && i < N) {
            const int64_t v = __ldg(idx + i);
            key[r] = expert_key(v, E);
            bad |= (key[r] < 0 && v != -1);
        }
    }
    if (bad) set_status(status, EP_ERR_BAD_EXPERT);
    int32_t* my = run + static_cast<int64_t>(warp) * E;
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        if (r < rounds) {
            const int k = key[r];
            const uint32_t peers = peers_of(k, kbits);
            if (k >= 0) rank[r] = my[k] + __popc(peers & lanemask_lt());
            __syncwarp();
            if (k >= 0 && lane == __ffs(peers) - 1) my[k] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();
    scan_across_warps(run, E, nwarps, tile_tot, 1);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r)
        if (r < rounds && key[r] >= 0) rank[r] += my[key[r]];
    cluster_barrier();  // every CTA's tile counts are complete

    // phase 2 (run[0 .. 2E) is free: ranks are in registers; tile_tot lies
    // beyond it because there are at least 4 warps)
    int32_t* tot = run;
    int32_t* base = run + E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const uint32_t local = smem_u32(tile_tot + e);
        int32_t c[CTAS];
#pragma unroll
        for (int q = 0; q < CTAS; ++q)
            c[q] = q < ntiles ? ld_cluster(cluster_map(local, static_cast<uint32_t>(q))) : 0;
        int32_t ts = 0, bs = 0;
#pragma unroll
        for (int q = 0; q < CTAS; ++q) {
            ts += c[q];
            bs += q < tile_id ? c[q] : 0;
        }
        tot[e] = ts;
        base[e] = bs;
    }
    cluster_barrier();  // no CTA reads another's shared memory after this

    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, per * static_cast<int>(threadIdx.x)), e1 = min(E, e0 + per);
    int64_t local = 0;
    for (int e = e0; e < e1; ++e) local += tot[e];
    int64_t total;
    int64_t off = block_exclusive_scan(local, &total);
    for (int e = e0; e < e1; ++e) {
        if (tile_id == 0) {
            offsets[e] = static_cast<int32_t>(off);
            counts[e] = tot[e];
        }
        base[e] += static_cast<int32_t>(off);
        off += tot[e];
    }
    if (tile_id == 0 && threadIdx.x == 0) offsets[E] = static_cast<int32_t>(total);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        const int64_t i = wbase + r * 32 + lane;
        if (r < rounds && i < N) slot[i] = key[r] >= 0 ? base[key[r]] + rank[r] : -1;
    }
}

// ---- single-launch layout (cooperative grid) -----------------------------------
// For tables of up to kCoopMaxTiles tiles, one cooperative launch does what
// the tile and finish kernels do, with one grid-wide barrier in between:
//   phase 1  per tile: ids, per-warp counts, ranks within the tile (kept in
//            registers), the tile's per-expert counts to tile_counts[tile][e]
//   phase 2  per tile: read the whole small [tiles][E] table (one coalesced,
//            batched pass), giving each expert's total and the rows taken by
//            earlier tiles; scan the totals across experts; write every
//            entry's final slot once. Block 0 writes counts and offsets.
// The barrier: each block publishes a 64-bit target value in its flag word
// and waits (bounded in time) until every block's flag holds it. The
// workspace starts with two words, an owner tag and a generation. Every
// process draws one random epoch in [2^63, 2^63 + 2^62) (top bit set, so no
// stale pair of 32-bit tile counts can spell a target). If the owner tag is
// this process's epoch, the target is the stored generation plus one;
// otherwise (a fresh or foreign workspace) it is the epoch plus one. Block 0
// stores the new generation and the owner tag once every block has passed
// the barrier (or, after a timed-out wait, the giving-up block does). So the
// barrier words need no clearing between calls, a replayed launch with
// identical arguments still waits for fresh flags, and within a process the
// targets only grow (2^62 calls before the counter could wrap), so no flag
// left by an earlier call, however long ago, can equal a later target.
__device__ __forceinline__ void st_release_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_acquire_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// All blocks of the grid arrive and wait; false (in every thread of the
// block) if some block's flag did not arrive within kWaitLimitNs.
__device__ bool grid_barrier(uint64_t* flags, int nblocks, uint64_t target) {
    __syncthreads();  // the block's writes precede thread 0's release (cumulative)
    if (threadIdx.x == 0) st_release_u64(flags + blockIdx.x, target);
    bool ok = true;
    for (int b = threadIdx.x; b < nblocks && ok; b += blockDim.x) {
        if (ld_acquire_u64(flags + b) == target) continue;
        const uint64_t t0 = global_timer_ns();
        while (ld_acquire_u64(flags + b) != target) {
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                ok = false;
                break;
            }
        }
    }
    return __syncthreads_and(ok) != 0;  // the acquires precede the block's reads
}

__global__ void __launch_bounds__(1024) layout_coop_kernel(const int64_t* __restrict__ idx, int64_t N, int E, int rounds,
                                   uint64_t* sync, int32_t* tile_counts, uint64_t epoch,
                                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                   int32_t* __restrict__ slot, int32_t* status) {
    extern __shared__ int32_t run[];  // [warps][E]; phase 2 reuses the first 2E words
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const int nt = gridDim.x, tile_id = blockIdx.x;
    const int64_t tile = static_cast<int64_t>(nwarps) * 32 * rounds;
    const int64_t wbase = tile * tile_id + static_cast<int64_t>(warp) * 32 * rounds;
    const int kbits = key_bits_for(E);

    griddep_launch_dependents();  // all blocks are resident (cooperative launch)
    // owner tag and generation: read before the barrier, replaced after it
    const uint64_t owner = reinterpret_cast<volatile uint64_t*>(sync)[0];
    const uint64_t g = reinterpret_cast<volatile uint64_t*>(sync)[1];
    const uint64_t g0 = (owner == epoch && g >= epoch) ? g : epoch;
    const uint64_t target = g0 + 1;

    // phase 1 ------------------------------------------------------------
    int key[kMaxRounds];
    int32_t rank[kMaxRounds];
    bool bad = false;
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        key[r] = -1;
        rank[r] = 0;
        const int64_t i = wbase + r * 32 + lane;
        if (r < rounds && i < N) {
            const int64_t v = __ldg(idx + i);
            key[r] = expert_key(v, E);
            bad |= (key[r] < 0 && v != -1);
        }
    }
    if (bad) set_status(status, EP_ERR_BAD_EXPERT);
    // one pass: each entry's rank among its warp's earlier entries of the
    // same expert, and the warp's per-expert counts
    int32_t* my = run + static_cast<int64_t>(warp) * E;
    for (int e = lane; e < E; e += 32) my[e] = 0;
    __syncwarp();
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        if (r < rounds) {
            const int k = key[r];
            const uint32_t peers = peers_of(k, kbits);
            if (k >= 0) rank[r] = my[k] + __popc(peers & lanemask_lt());
            __syncwarp();
            if (k >= 0 && lane == __ffs(peers) - 1) my[k] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();
    // counts -> each warp's first rank within the tile; tile totals published
    scan_across_warps(run, E, nwarps, tile_counts + static_cast<int64_t>(tile_id) * E, 1);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r)
        if (r < rounds && key[r] >= 0) rank[r] += my[key[r]];
    if (!grid_barrier(sync + 2, nt, target)) {
        // leave the generation past every flag this call may have published
        if (threadIdx.x == 0) {
            set_status(status, EP_ERR_TIMEOUT);
            st_release_u64(sync + 1, target);
            st_release_u64(sync, epoch);
        }
        return;
    }
    if (tile_id == 0 && threadIdx.x == 0) {
        st_release_u64(sync + 1, target);
        st_release_u64(sync, epoch);
    }

    // phase 2: per expert, its total and the rows of earlier tiles. Q threads
    // share an expert (tiles q, q+Q, ...), each with all its loads in flight
    // at once; partial sums go to shared memory and one thread per expert
    // adds them up. No atomics.
    __syncthreads();
    const int Q = max(1, min(static_cast<int>(blockDim.x) / E, nwarps / 2));
    int32_t* part_t = run;                              // [Q][E] totals
    int32_t* part_b = run + static_cast<int64_t>(Q) * E;  // [Q][E] earlier tiles
    for (int x = threadIdx.x; x < E * Q; x += blockDim.x) {
        const int e = x % E, q = x / E;
        int32_t t_sum = 0, b_sum = 0;
        for (int t0 = q; t0 < nt; t0 += 16 * Q) {
            int32_t c[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const int t = t0 + u * Q;
                c[u] = t < nt ? __ldcg(tile_counts + static_cast<int64_t>(t) * E + e) : 0;
            }
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                t_sum += c[u];
                b_sum += (t0 + u * Q < tile_id) ? c[u] : 0;
            }
        }
        part_t[static_cast<int64_t>(q) * E + e] = t_sum;
        part_b[static_cast<int64_t>(q) * E + e] = b_sum;
    }
    __syncthreads();
    int32_t* tot = part_t;   // row 0 receives the sums
    int32_t* base = part_b;
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, per * static_cast<int>(threadIdx.x)), e1 = min(E, e0 + per);
    int64_t local = 0;
    for (int e = e0; e < e1; ++e) {
        int32_t ts = 0, bs = 0;
        for (int q = 0; q < Q; ++q) {
            ts += part_t[static_cast<int64_t>(q) * E + e];
            bs += part_b[static_cast<int64_t>(q) * E + e];
        }
        tot[e] = ts;
        base[e] = bs;
        local += ts;
    }
    int64_t total;
    int64_t off = block_exclusive_scan(local, &total);
    for (int e = e0; e < e1; ++e) {
        if (tile_id == 0) {
            offsets[e] = static_cast<int32_t>(off);
            counts[e] = tot[e];
        }
        base[e] += static_cast<int32_t>(off);
        off += tot[e];
    }
    if (tile_id == 0 && threadIdx.x == 0) offsets[E] = static_cast<int32_t>(total);
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kMaxRounds; ++r) {
        const int64_t i = wbase + r * 32 + lane;
        if (r < rounds && i < N) slot[i] = key[r] >= 0 ? base[key[r]] + rank[r] : -1;
    }
}

}  // namespace

LayoutPlan plan_layout(int64_t N, int E) {
    LayoutPlan p{};
    int warps = static_cast<int>(kRunSmemBudget / (sizeof(int32_t) * static_cast<size_t>(E)));
    warps = warps < 1 ? 1 : (warps > 32 ? 32 : warps);
    p.warps = warps;
    const int64_t per_round = 32LL * warps;  // entries per round of the whole block
    if (N <= per_round * kFusedRounds) {
        // one block: as few warps as give each about kSingleRounds rounds
        p.num_tiles = 1;
        int64_t w = (N + 32LL * kSingleRounds - 1) / (32LL * kSingleRounds);
        w = w < 1 ? 1 : (w > warps ? warps : w);
        warps = static_cast<int>(w);
        p.warps = warps;
        const int64_t pr = 32LL * warps;
        p.rounds = static_cast<int>((N + pr - 1) / pr);
        if (p.rounds < 1) p.rounds = 1;
        p.tile = pr * p.rounds;
        p.smem = sizeof(int32_t) * static_cast<size_t>(E) * warps;
        return p;
    } else {
        int64_t r = (N + per_round * kTargetTiles - 1) / (per_round * kTargetTiles);
        p.rounds = static_cast<int>(r < 1 ? 1 : (r > kMaxRounds ? kMaxRounds : r));
    }
    p.tile = per_round * p.rounds;
    p.num_tiles = static_cast<int>((N + p.tile - 1) / p.tile);
    p.smem = sizeof(int32_t) * static_cast<size_t>(E) * warps;
    // one cluster when the table fits kClusterCtas tiles of <= 8 rounds
    p.cluster = p.num_tiles > 1 && N <= per_round * kClusterCtas * kMaxRounds;
    if (p.cluster) {
        p.rounds = static_cast<int>((N + per_round * kClusterCtas - 1) / (per_round * kClusterCtas));
        p.tile = per_round * p.rounds;
        p.num_tiles = static_cast<int>((N + p.tile - 1) / p.tile);
        p.smem = sizeof(int32_t) * static_cast<size_t>(E) * (warps + 1);
        p.workspace_bytes = 0;
        p.coop = false;
        return p;
    }
    p.coop = p.num_tiles > 1 && p.num_tiles <= kCoopMaxTiles;
    if (p.num_tiles > 1) {
        // [owner][generation][flag x tiles] | tile_counts[tiles][E]
        auto up16 = [](size_t v) { return (v + 15) & ~static_cast<size_t>(15); };
        p.counts_off = up16(sizeof(uint64_t) * (2 + static_cast<size_t>(p.num_tiles)));
        p.workspace_bytes = p.counts_off + sizeof(int32_t) * static_cast<size_t>(E) * p.num_tiles;
    }
    return p;
}

bool plan_layout_wide_cluster(int64_t N, int E, LayoutPlan* out) {
    LayoutPlan p = plan_layout(N, E);
    const int64_t per_round = 32LL * p.warps;
    if (p.workspace_bytes == 0 || N > per_round * kWideClusterCtas * kMaxRounds) return false;
    p.rounds = static_cast<int>((N + per_round * kWideClusterCtas - 1) /
                                (per_round * kWideClusterCtas));
    p.tile = per_round * p.rounds;
    p.num_tiles = static_cast<int>((N + p.tile - 1) / p.tile);
    if (p.num_tiles <= kClusterCtas || p.num_tiles > kWideClusterCtas) return false;
    p.smem = sizeof(int32_t) * static_cast<size_t>(E) * (p.warps + 1);
    p.cluster = true;
    p.coop = false;
    p.counts_off = 0;
    p.workspace_bytes = 0;
    // only where this GPU can hold such a cluster at all
    auto kern = layout_cluster_kernel<kWideClusterCtas>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(p.smem)) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(p.num_tiles));
    cfg.blockDim = dim3(static_cast<unsigned>(p.warps * 32));
    cfg.dynamicSmemBytes = p.smem;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = static_cast<unsigned>(p.num_tiles);
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess || clusters < 1) {
        (void)cudaGetLastError();
        return false;
    }
    *out = p;
    return true;
}

namespace {
// Per-process epoch of the layout barriers' generation values: random, in
// [2^63, 2^63 + 2^62).
uint64_t barrier_epoch() {
    static const uint64_t epoch = [] {
        const uint64_t t = static_cast<uint64_t>(
            std::chrono::steady_clock::now().time_since_epoch().count());
        uint64_t h = t ^ (static_cast<uint64_t>(getpid()) << 21);
        // splitmix64 finaliser: spreads the clock and pid bits over the word
        h ^= h >> 30;
        h *= 0xBF58476D1CE4E5B9ull;
        h ^= h >> 27;
        h *= 0x94D049BB133111EBull;
        h ^= h >> 31;
        return (uint64_t{1} << 63) | (h & ((uint64_t{1} << 62) - 1));
    }();
    return epoch;
}
}  // namespace

cudaError_t launch_layout(const int64_t* idx, int64_t N, int E, int32_t* counts,
                          int32_t* offsets, int32_t* slot, void* workspace,
                          const LayoutPlan& p, int32_t* status, cudaStream_t stream) {
    const int threads = p.warps * 32;
    if (p.num_tiles == 1) {
        // The tile kernel's dynamic shared memory can exceed the default 48 KB
        // (it also holds a few static words for the block scan).
        cudaError_t err = cudaFuncSetAttribute(layout_tile_kernel<true>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kRunSmemBudget));
        if (err != cudaSuccess) return err;
        return launch_dependent(layout_tile_kernel<true>, 1, threads, p.smem, stream, idx, N, E,
                                p.rounds, 1, static_cast<int32_t*>(nullptr), counts, offsets,
                                slot, status);
    }
    if (p.cluster) {
        const bool wide = p.num_tiles > kClusterCtas;
        auto kern = wide ? layout_cluster_kernel<kWideClusterCtas> : layout_cluster_kernel<kClusterCtas>;
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(p.smem));
        if (err != cudaSuccess) return err;
        if (wide &&
            (err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) !=
                cudaSuccess)
            return err;
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(p.num_tiles));
        cfg.blockDim = dim3(static_cast<unsigned>(threads));
        cfg.dynamicSmemBytes = p.smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2]{};
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(p.num_tiles);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        // as launch_dependent: may start while the previous kernel finishes
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = launch_overlap_allowed(stream) ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        return cudaLaunchKernelEx(&cfg, kern, idx, N, E, p.rounds, counts, offsets, slot, status);
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint64_t* sync = reinterpret_cast<uint64_t*>(ws);
    int32_t* tile_counts = reinterpret_cast<int32_t*>(ws + p.counts_off);
    if (p.coop) {
        cudaError_t err = cudaFuncSetAttribute(layout_coop_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(kRunSmemBudget));
        if (err != cudaSuccess) return err;
        int rounds = p.rounds;
        uint64_t epoch = barrier_epoch();
        void* args[] = {(void*)&idx,  (void*)&N,      (void*)&E,       (void*)&rounds,
                        (void*)&sync, (void*)&tile_counts, (void*)&epoch, (void*)&counts,
                        (void*)&offsets, (void*)&slot, (void*)&status};
        err = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(layout_coop_kernel),
                                          dim3(p.num_tiles), dim3(threads), args, p.smem, stream);
        if (err == cudaSuccess) return cudaSuccess;
        if (err != cudaErrorCooperativeLaunchTooLarge) return err;
        (void)cudaGetLastError();  // too many tiles to be resident at once: two launches instead
    }
    cudaError_t err = cudaFuncSetAttribute(layout_tile_kernel<false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kRunSmemBudget));
    if (err != cudaSuccess) return err;
    err = launch_dependent(layout_tile_kernel<false>, p.num_tiles, threads, p.smem, stream, idx, N,
                           E, p.rounds, p.num_tiles, tile_counts, counts, offsets, slot, status);
    if (err != cudaSuccess) return err;
    if (p.num_tiles <= kMaxRedundantTiles)
        return launch_dependent(layout_finish_kernel<false>, p.num_tiles, kFinishThreads,
                                2 * sizeof(int32_t) * E, stream,
                                static_cast<const int32_t*>(tile_counts), p.num_tiles, E, N, p.tile,
                                counts, offsets, slot);
    err = launch_dependent(layout_scan_kernel, 1, kScanThreads, 0, stream, tile_counts,
                           p.num_tiles, E, counts, offsets);
    if (err != cudaSuccess) return err;
    return launch_dependent(layout_finish_kernel<true>, p.num_tiles, kFinishThreads,
                            sizeof(int32_t) * E, stream, static_cast<const int32_t*>(tile_counts),
                            p.num_tiles, E, N, p.tile, counts, offsets, slot);
}

}  // namespace ep
