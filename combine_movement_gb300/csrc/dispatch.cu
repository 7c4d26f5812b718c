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
#include "routing.cuh"
#include "work_split.cuh"

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
#ifndef EP_DISPATCH_STORE_FIRST
#define EP_DISPATCH_STORE_FIRST 0
#endif
#ifndef EP_DISPATCH_LOAD_NORMAL
#define EP_DISPATCH_LOAD_NORMAL 0
#endif
#ifndef EP_DISPATCH_FILL_RING
#define EP_DISPATCH_FILL_RING 1
#endif
#ifndef EP_DISPATCH_L2_PREFETCH
#define EP_DISPATCH_L2_PREFETCH 1
#endif
#ifndef EP_DISPATCH_L2_TAIL
#define EP_DISPATCH_L2_TAIL 1
#endif

constexpr unsigned kFullMask = 0xFFFFFFFFu;
constexpr int kDispatchWarps = EP_DISPATCH_WARPS;
// Units beyond the filled ring that a warp prefetches into L2 while the
// layout holds back its first store (full budget only).
#ifndef EP_DISPATCH_L2_UNITS
#define EP_DISPATCH_L2_UNITS 4
#endif
constexpr int64_t kL2PrefetchUnits = EP_DISPATCH_L2_UNITS;

// Bytes reserved in front of the stages for the mbarriers (8 B per stage per
// warp), rounded up so every stage starts 128-byte aligned.
__host__ __device__ constexpr uint32_t barrier_region(int stages, int warps) {
    return (8u * stages * warps + 127u) & ~127u;
}

// Entries [i0, i1) of the routing table: the (token, k) cells of the tokens
// a fused-kernel CTA moves (the union of its warps' unit ranges).
struct CtaEntries {
    int64_t i0, i1;
};
__device__ __forceinline__ CtaEntries cta_entries(const DispatchArgs& a, int64_t units,
                                                  int64_t nw_total) {
    const int nwarps = blockDim.x >> 5;
    const int64_t cu0 = split_begin(units, static_cast<int64_t>(blockIdx.x) * nwarps, nw_total);
    const int64_t cu1 = split_begin(units, static_cast<int64_t>(blockIdx.x + 1) * nwarps, nw_total);
    const int64_t t0 = div_floor(cu0, a.n_chunks);
    const int64_t t1 = cu1 > cu0 ? div_floor(cu1 - 1, a.n_chunks) + 1 : t0;
    return {t0 * a.K, t1 * a.K};
}

// Layout prologue of the fused kernel (see dispatch_kernel). All threads of
// the CTA take part; ends with a block barrier after which the slots of the
// CTA's entries are in global memory and, when f.own_off != 0, in shared
// memory too (own_slot[i - i0]). `prefetch()` runs once, right after the
// first routing-table loads are issued: the ring's first row loads then
// queue behind them instead of delaying them.
template <class Prefetch>
__device__ __forceinline__ void fused_layout(const DispatchArgs& a, const FusedLayoutArgs& f,
                                          uint8_t* smem, CtaEntries own, Prefetch prefetch) {
    const int E = f.E;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t* total = reinterpret_cast<int32_t*>(smem + f.hist_off);
    int32_t* run = total + E;
    int16_t* own_key = reinterpret_cast<int16_t*>(smem + f.own_off);
    int32_t* own_slot = reinterpret_cast<int32_t*>(smem + f.own_off + kFusedOwnCap * sizeof(int16_t));
    const bool keep = f.own_off != 0;
    const int64_t N = a.T * a.K;
    const int64_t i0 = own.i0, i1 = own.i1;

    for (int e = threadIdx.x; e < E; e += blockDim.x) total[e] = run[e] = 0;
    __syncthreads();
    bool bad = false;
    auto count = [&](int64_t i, int64_t v) {
        const int e = expert_key(v, E);
        if (e >= 0) {
            atomicAdd(&total[e], 1);
            if (i < i0) atomicAdd(&run[e], 1);
        } else if (v != -1) {
            bad = true;
        }
        // the CTA's own entries are ranked from shared memory below
        if (keep && i >= i0 && i < i1) own_key[i - i0] = static_cast<int16_t>(e);
    };
    // 16-byte loads (two ids each), 16 in flight per thread; an 8-byte-
    // aligned first id and an odd last id are read on their own. The trip
    // count is the same for every lane of a warp (w0 is the warp's first
    // lane), so prefetch() and its bulk copies always run in a converged
    // warp, as in the ring: a warp split by a per-lane bound faulted with a
    // misaligned address on its first bulk loads (150 ids on one CTA).
    const int64_t head = (reinterpret_cast<uintptr_t>(f.idx) & 15u) ? 1 : 0;
    const int64_t pairs = N > head ? (N - head) / 2 : 0;
    const longlong2* pv = reinterpret_cast<const longlong2*>(f.idx + head);
    constexpr int kBatch = 16;
    bool prefetched = false;
    for (int64_t w0 = threadIdx.x & ~31u; w0 < pairs;
         w0 += static_cast<int64_t>(blockDim.x) * kBatch) {
        const int64_t b0 = w0 + lane;
        longlong2 v[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int64_t q = b0 + static_cast<int64_t>(u) * blockDim.x;
            v[u] = q < pairs ? __ldg(pv + q) : make_longlong2(-1, -1);
        }
        __syncwarp();
        if (!prefetched) {
            prefetch();
            prefetched = true;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int64_t q = b0 + static_cast<int64_t>(u) * blockDim.x;
            if (q < pairs) {
                count(head + 2 * q, v[u].x);
                count(head + 2 * q + 1, v[u].y);
            }
        }
    }
    __syncwarp();
    if (!prefetched) prefetch();
    if (threadIdx.x == 0) {
        if (head && N > 0) count(0, __ldg(f.idx));
        const int64_t last = head + 2 * pairs;
        if (last < N) count(last, __ldg(f.idx + last));
    }
    if (bad) set_status(a.status, EP_ERR_BAD_EXPERT);
    __syncthreads();
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int e0 = min(E, per * static_cast<int>(threadIdx.x)), e1 = min(E, e0 + per);
    int64_t local = 0;
    for (int e = e0; e < e1; ++e) local += total[e];
    int64_t all;
    int64_t off = block_exclusive_scan(local, &all);
    for (int e = e0; e < e1; ++e) {
        if (blockIdx.x == 0) {
            f.offsets[e] = static_cast<int32_t>(off);
            f.counts[e] = total[e];
        }
        run[e] += static_cast<int32_t>(off);
        off += total[e];
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) f.offsets[E] = static_cast<int32_t>(all);
    __syncthreads();
    if (warp == 0) {
        // 8 rounds of ids are read together (from shared memory when kept
        // there, else one global-memory latency per 256 entries), then
        // ranked round by round in entry order.
        const int kbits = key_bits_for(E);
        constexpr int kRounds = 8;
        for (int64_t b0 = i0; b0 < i1; b0 += 32 * kRounds) {
            int key[kRounds];
#pragma unroll
            for (int r = 0; r < kRounds; ++r) {
                const int64_t i = b0 + r * 32 + lane;
                key[r] = i >= i1 ? -1 : keep ? own_key[i - i0] : expert_key(__ldg(f.idx + i), E);
            }
#pragma unroll
            for (int r = 0; r < kRounds; ++r) {
                const int64_t i = b0 + r * 32 + lane;
                if (b0 + r * 32 >= i1) break;
                const uint32_t peers = peers_of(key[r], kbits);
                if (i < i1) {
                    const int32_t sl = key[r] >= 0 ? run[key[r]] + __popc(peers & lanemask_lt()) : -1;
                    f.slot[i] = sl;
                    if (keep) own_slot[i - i0] = sl;
                }
                __syncwarp();
                if (key[r] >= 0 && lane == __ffs(peers) - 1) run[key[r]] += __popc(peers);
                __syncwarp();
            }
        }
    }
    __syncthreads();
}

// Plain (coherent) 32-bit load, for slots written earlier in the same kernel.
__device__ __forceinline__ int32_t ld_plain_s32(const int32_t* p) {
    int32_t v;
    asm volatile("ld.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// FUSED: layout computed by every CTA for its own tokens before its ring
// (ep_layout_dispatch). Each CTA reads the whole routing table once (it is
// small next to the rows), keeping in shared memory each expert's total and
// the number of entries before the CTA's first token; a scan across experts
// gives each expert's first row; warp 0 then ranks the CTA's own entries in
// entry order (per-bit ballot peer groups) and writes their slots. No CTA
// waits on another and no workspace is needed. Block 0 writes counts and
// offsets; a token split between two CTAs gets the same slots from both.
template <int NS, int P, bool FUSED>
__global__ void __launch_bounds__(kDispatchWarps * 32, 1)
    dispatch_kernel(const DispatchArgs a, const FusedLayoutArgs f) {
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

    // this launch's units, split evenly over its warps
    const int64_t units = a.unit_count;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * nwarps + warp;
    const int64_t nw_total = static_cast<int64_t>(gridDim.x) * nwarps;
    const int64_t u0 = a.unit_base + split_begin(units, gw, nw_total);
    const int64_t n = a.unit_base + split_begin(units, gw + 1, nw_total) - u0;

    // L2 policies: x is read once (evict first); the receive rows are
    // written once and next read by the experts (normal).
#if EP_DISPATCH_STORE_FIRST
    const uint64_t pol_store = policy_evict_first();
#else
    const uint64_t pol_store = policy_evict_normal();
#endif
#if EP_DISPATCH_LOAD_NORMAL
    const uint64_t pol_load = policy_evict_normal();
#else
    const uint64_t pol_load = policy_evict_first();
#endif

    // Bulk-load the next unit (token lt, chunk lc) into the stage of local
    // unit j (units are loaded in order, so (lt, lc) just advances).
    int64_t lt = div_floor(u0, a.n_chunks);
    uint32_t lc = static_cast<uint32_t>(u0 - lt * a.n_chunks);
    auto issue_load = [&](int64_t j) {
        const int64_t t = lt;
        const uint32_t c = lc;
        if (++lc == a.n_chunks) {
            lc = 0;
            ++lt;
        }
        if (!leader) return;
        const uint32_t off = c * a.chunk_bytes;
        const uint32_t bytes = min(a.chunk_bytes, a.row_bytes - off);
        const int s = static_cast<int>(j % NS);
        const uint32_t bar = bar0 + 8u * s;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_load(buf0 + static_cast<uint32_t>(s) * a.stage_bytes,
                  a.x + t * static_cast<int64_t>(a.row_bytes) + off, bytes, bar, pol_load);
    };

    // With a.tail_l2_prefetch, each warp also brings its share of the rows
    // of the tail launch that follows (DispatchArgs::tail_units) into L2
    // while the layout holds back its first store: the tail's CTAs start
    // late, when HBM is busy with the ring's stores.
    auto prefetch_tail_rows = [&](uint64_t policy) {
        if (!EP_DISPATCH_L2_TAIL || !a.tail_l2_prefetch || a.tail_units <= 0) return;
        const int64_t tb = a.unit_base + a.unit_count;
        const int64_t q1 = tb + split_begin(a.tail_units, gw + 1, nw_total);
        for (int64_t q = tb + split_begin(a.tail_units, gw, nw_total); q < q1; ++q) {
            const int64_t qt = div_floor(q, a.n_chunks);
            const uint32_t off = static_cast<uint32_t>(q - qt * a.n_chunks) * a.chunk_bytes;
            bulk_prefetch_l2(a.x + qt * static_cast<int64_t>(a.row_bytes) + off,
                             min(a.chunk_bytes, a.row_bytes - off), policy);
        }
    };

    // Loads issued before the ring starts: P, or the whole ring (NS) when
    // the kernel has to wait before its first store anyway (the fused
    // layout, or a layout kernel it overlaps) and no stage is being stored.
    const bool fill_ring = EP_DISPATCH_FILL_RING && (FUSED || a.x_ready != 0);
    const int64_t prefilled = fill_ring ? (n < NS ? n : NS) : (n < P ? n : P);
    auto first_loads = [&]() {
        for (int64_t j = 0; j < prefilled; ++j) issue_load(j);
#if EP_DISPATCH_L2_PREFETCH
        // While the layout still holds back the first store, the warp's
        // next kL2PrefetchUnits rows are brought into L2 too (evict-last, so
        // the receive rows streaming through L2 do not push them out
        // first). More than that crowds L2 for the rest of the kernel.
        if (fill_ring && leader && a.l2_prefetch != 0) {
            const uint64_t pol_keep = policy_evict_last();
            int64_t pt = lt;
            uint32_t pc = lc;
            const int64_t end = n < prefilled + kL2PrefetchUnits ? n : prefilled + kL2PrefetchUnits;
            for (int64_t j = prefilled; j < end; ++j) {
                const uint32_t off = pc * a.chunk_bytes;
                bulk_prefetch_l2(a.x + pt * static_cast<int64_t>(a.row_bytes) + off,
                                 min(a.chunk_bytes, a.row_bytes - off), pol_keep);
                if (++pc == a.n_chunks) {
                    pc = 0;
                    ++pt;
                }
            }
            prefetch_tail_rows(pol_keep);
        }
#endif
    };
    // Every global-memory access waits for the previous kernel on the stream
    // (programmatic dependent launch), except the first row loads when x is
    // known to be complete already (a.x_ready: the layout kernel of
    // ep_layout_dispatch precedes this launch); they then overlap it.
    const bool early = !FUSED && a.x_ready != 0;
    if (early) first_loads();
#if EP_DISPATCH_L2_PREFETCH
    // Without x_ready the kernel before this one may still be writing x, so
    // nothing may be copied into shared memory yet; bringing the first
    // rows into L2 is safe (L2 is coherent: a later write updates the
    // line) and uses the time this kernel would otherwise only wait.
    if (!FUSED && !early && a.l2_prefetch != 0 && leader) {
        const uint64_t pol_keep = policy_evict_last();
        int64_t pt = lt;
        uint32_t pc = lc;
        const int64_t end = n < prefilled + kL2PrefetchUnits ? n : prefilled + kL2PrefetchUnits;
        for (int64_t j = 0; j < end; ++j) {
            const uint32_t off = pc * a.chunk_bytes;
            bulk_prefetch_l2(a.x + pt * static_cast<int64_t>(a.row_bytes) + off,
                             min(a.chunk_bytes, a.row_bytes - off), pol_keep);
            if (++pc == a.n_chunks) {
                pc = 0;
                ++pt;
            }
        }
    }
#endif
    // (A tail launch's CTAs skip the wait, all but its last; see
    // DispatchArgs::tail.)
    if (!a.tail || blockIdx.x == gridDim.x - 1) griddep_wait();
    griddep_launch_dependents();

    // The fused kernel's entries: the CTA's slots stay in shared memory
    // (own_slot) when f.own_off != 0.
    const CtaEntries own = FUSED ? cta_entries(a, units, nw_total) : CtaEntries{0, 0};
    const int32_t* own_slot =
        reinterpret_cast<const int32_t*>(smem + f.own_off + kFusedOwnCap * sizeof(int16_t));

    // Lanes k < K hold slot[t][k] (and topk_w[t][k]) of the current token and
    // of the next one, loaded a token ahead.
    auto load_slot = [&](int64_t t) -> int32_t {
        if (t >= a.T || lane >= a.K) return -1;
        if (!FUSED) return __ldg(a.slot + t * a.K + lane);
        const int64_t i = t * a.K + lane;
        if (f.own_off != 0) return (i >= own.i0 && i < own.i1) ? own_slot[i - own.i0] : -1;
        return ld_plain_s32(a.slot + i);
    };
    auto load_w = [&](int64_t t) -> float {
        return (a.topk_w != nullptr && t < a.T && lane < a.K) ? __ldg(a.topk_w + t * a.K + lane)
                                                              : 0.0f;
    };

    // The rows of x do not depend on the layout, so the first loads go out
    // before the fused kernel computes it, right behind its routing-table
    // loads (every thread of the CTA then takes part in the layout, whatever
    // its own share of units).
    if (FUSED)
        fused_layout(a, f, smem, own, first_loads);
    else if (!early)
        first_loads();
    if (n <= 0) return;

    int64_t tok = div_floor(u0, a.n_chunks);
    int32_t s_cur = load_slot(tok), s_next = load_slot(tok + 1);
    float w_cur = load_w(tok), w_next = load_w(tok + 1);

    // (token, chunk) of local unit j, advanced without divisions
    int64_t t = tok;
    uint32_t c = static_cast<uint32_t>(u0 - tok * a.n_chunks);
    for (int64_t j = 0; j < n; ++j, ++c) {
        if (c == a.n_chunks) {
            c = 0;
            ++t;
        }
        if (t != tok) {
            tok = t;
            s_cur = s_next;
            w_cur = w_next;
            s_next = load_slot(t + 1);
            w_next = load_w(t + 1);
        }

        // Refill: the stage of unit j+P was last used by unit j+P-NS; its
        // stores must have finished reading shared memory.
        if (j + P < n && j + P >= prefilled) {
            if (leader) bulk_wait_read<NS - P - 1>();
            issue_load(j + P);
        }

        const int s = static_cast<int>(j % NS);
        uint32_t ok = 1;
        if (leader) ok = mbar_wait_bounded(bar0 + 8u * s, static_cast<uint32_t>((j / NS) & 1));
        ok = __shfl_sync(kFullMask, ok, leader_lane);
        if (!ok) {
            if (leader) {
                set_status(a.status, EP_ERR_TIMEOUT);
                const int64_t last_issued = (j + P < n ? j + P : n - 1) > prefilled - 1
                                                ? (j + P < n ? j + P : n - 1)
                                                : prefilled - 1;
                mbar_drain_bounded<NS>(bar0, j, last_issued);
            }
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
    // Shared memory must outlive every bulk store that reads it: wait until
    // they have all read their stage. Their writes to global memory need no
    // wait here (they complete with the grid, before any later kernel on the
    // stream, or one waiting on this grid's completion, can see the grid
    // done), so the CTA leaves without the write acknowledgements' latency.
    if (leader) bulk_wait_read<0>();
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
    const int64_t u0 = split_begin(units, gw, nw_total), u1 = split_begin(units, gw + 1, nw_total);
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
// While launches overlap (full SM budget) the ring has one stage fewer: a
// dispatch CTA then takes 172 KB of shared memory instead of 229 KB, so the
// SM does not have to switch to its largest shared-memory configuration
// (the least L1) for dispatch. With the kernels overlapping that made the
// DeepSeek-V3 prefill step 192.8 -> 181.0 us (T=16384: 746 -> 695 us);
// other shapes and decode were unchanged. Forcing the largest configuration
// on every kernel brought the step back to 191.4 us, and any ring under
// ~190 KB (6 warps x 4 stages, or 3.5 KB chunks) gave the same gain. Below
// the full budget launches do not overlap and the 4-stage ring is as fast
// or up to 2.5 % faster.
#ifndef EP_DISPATCH_SHARED_STAGES
#define EP_DISPATCH_SHARED_STAGES 3
#endif
constexpr int kSharedStages = EP_DISPATCH_SHARED_STAGES;
static_assert(kSharedStages > kPrefetch, "need more stages than loads in flight");
// Warps of a tail CTA (DispatchArgs::tail_units), one unit each: 2 where
// rows are cut into chunks, 4 where a row is one chunk. Measured with the
// combine that follows (step back to back): DeepSeek-V3 prefill (two 7 KB
// chunks per row) 162.8 / 165.3 / 174.1 us with 2 / 3 / 4 warps, skewed
// Zipf (8 KB rows, one chunk) 157.3 / 146.6 / 145.9 us with 2 / 3 / 4.
#ifndef EP_DISPATCH_TAIL_WARPS
#define EP_DISPATCH_TAIL_WARPS 0
#endif
int tail_warps(const DispatchArgs& a) {
    if (EP_DISPATCH_TAIL_WARPS > 0) return EP_DISPATCH_TAIL_WARPS;
    return a.n_chunks >= 2 ? 2 : 4;
}
// 1: a tail CTA asks for more shared memory than an SM has beside a ring
// CTA, so it never shares an SM with one.
#ifndef EP_DISPATCH_TAIL_EXCLUSIVE
#define EP_DISPATCH_TAIL_EXCLUSIVE 1
#endif

}  // namespace

template <int NS>
cudaError_t launch_ring(const DispatchArgs& a, int num_sms, cudaStream_t stream) {
    const size_t smem = static_cast<size_t>(barrier_region(NS, kDispatchWarps)) +
                        static_cast<size_t>(kDispatchWarps) * NS * a.stage_bytes;
    const size_t request = smem < kExclusiveSmem ? kExclusiveSmem : smem;
    auto kern = dispatch_kernel<NS, kPrefetch, false>;
    cudaError_t err =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(request));
    if (err != cudaSuccess) return err;
    DispatchArgs ring = a;
    ring.unit_count = a.unit_count - a.tail_units;
    const int64_t ctas_needed = (ring.unit_count + kDispatchWarps - 1) / kDispatchWarps;
    const int grid = static_cast<int>(ctas_needed < num_sms ? ctas_needed : num_sms);
    if (grid <= 0) return cudaSuccess;
    err = launch_dependent(kern, grid, kDispatchWarps * 32, request, stream, ring, FusedLayoutArgs{});
    if (err != cudaSuccess || a.tail_units <= 0) return err;
    // The tail: small CTAs of tw warps, one unit per warp, on the
    // same ring shape, each asking for more shared memory than an SM has
    // beside a ring CTA (DispatchArgs::tail_units).
    const int tw = tail_warps(a);
    DispatchArgs tail = a;
    tail.unit_base = a.unit_base + ring.unit_count;
    tail.unit_count = a.tail_units;
    tail.tail = 1;
    tail.x_ready = 0;
    tail.l2_prefetch = 0;
    tail.tail_l2_prefetch = 0;
    int dev = 0, per_sm = 0, reserved = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    if ((err = cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
        cudaSuccess)
        return err;
    if ((err = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) !=
        cudaSuccess)
        return err;
    const size_t need = static_cast<size_t>(barrier_region(NS, tw)) +
                        static_cast<size_t>(tw) * NS * a.stage_bytes;
    // free beside a ring CTA, less the tail CTA's own reserved bytes
    const long long spare = static_cast<long long>(per_sm) - static_cast<long long>(request) -
                            2ll * reserved;
    size_t tail_request = need;
    if (EP_DISPATCH_TAIL_EXCLUSIVE && spare >= 0 && static_cast<size_t>(spare) + 128 > tail_request)
        tail_request = (static_cast<size_t>(spare) + 128) & ~static_cast<size_t>(127);
    auto tkern = dispatch_kernel<NS, kPrefetch, false>;
    if (tail_request > request &&
        (err = cudaFuncSetAttribute(tkern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(tail_request))) != cudaSuccess)
        return err;
    const int tail_grid = static_cast<int>((a.tail_units + tw - 1) / tw);
    return launch_dependent(tkern, tail_grid, tw * 32, tail_request, stream, tail,
                            FusedLayoutArgs{});
}

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
    // the ring the rows were planned for
    if (a.ring_stages == kSharedStages) return launch_ring<kSharedStages>(a, num_sms, stream);
    if (a.ring_stages != kStages) return cudaErrorInvalidValue;
    return launch_ring<kStages>(a, num_sms, stream);
}

int dispatch_ring_stages(bool fused, cudaStream_t stream) {
    // whenever launches may overlap, in an SM partition too: there the
    // 4-stage ring made the prefill step 34-40 % slower at 16-48 SMs
    return (!fused && launch_overlap_allowed(stream)) ? kSharedStages : kStages;
}

// Stage size the host plans rows with: the per-warp slice (what is left of
// the opt-in limit after `reserve` bytes) split into the ring's `stages`
// stages, rounded down to 16 bytes.
uint32_t dispatch_stage_capacity(int smem_optin, size_t reserve, int stages) {
    const size_t avail = static_cast<size_t>(smem_optin) - barrier_region(stages, kDispatchWarps);
    if (avail <= reserve) return 0;
    const size_t per_warp = (avail - reserve) / kDispatchWarps;
    return static_cast<uint32_t>((per_warp / stages) & ~static_cast<size_t>(15));
}

int dispatch_warps() { return kDispatchWarps; }

cudaError_t launch_layout_dispatch(const DispatchArgs& a, FusedLayoutArgs f, int num_sms,
                                   cudaStream_t stream) {
    if (a.ring_stages != kStages) return cudaErrorInvalidValue;
    const size_t ring = static_cast<size_t>(barrier_region(kStages, kDispatchWarps)) +
                        static_cast<size_t>(kDispatchWarps) * kStages * a.stage_bytes;
    f.hist_off = static_cast<uint32_t>(ring);
    const size_t hist_end = ring + 2 * sizeof(int32_t) * static_cast<size_t>(f.E);
    const int64_t units = a.T * static_cast<int64_t>(a.n_chunks);
    const int64_t ctas_needed = (units + kDispatchWarps - 1) / kDispatchWarps;
    const int grid = static_cast<int>(ctas_needed < num_sms ? ctas_needed : num_sms);
    // the most entries any CTA lays out (same split as the kernel's)
    int64_t most = 0;
    const int64_t nw_total = static_cast<int64_t>(grid > 0 ? grid : 1) * kDispatchWarps;
    for (int b = 0; b < grid; ++b) {
        const int64_t cu0 = units * (static_cast<int64_t>(b) * kDispatchWarps) / nw_total;
        const int64_t cu1 = units * (static_cast<int64_t>(b + 1) * kDispatchWarps) / nw_total;
        const int64_t t0 = cu0 / a.n_chunks;
        const int64_t t1 = cu1 > cu0 ? (cu1 - 1) / a.n_chunks + 1 : t0;
        if ((t1 - t0) * a.K > most) most = (t1 - t0) * a.K;
    }
    f.own_off = most <= kFusedOwnCap ? static_cast<uint32_t>((hist_end + 15) & ~size_t{15}) : 0u;
    size_t smem = ((hist_end + 15) & ~size_t{15}) + kFusedOwnBytes;
    if (smem < kExclusiveSmem) smem = kExclusiveSmem;
    auto kern = dispatch_kernel<kStages, kPrefetch, true>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(smem));
    if (err != cudaSuccess) return err;
    return launch_dependent(kern, grid > 0 ? grid : 1, kDispatchWarps * 32, smem, stream, a, f);
}

}  // namespace ep
