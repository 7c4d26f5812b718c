// ep_api.cu -- the C ABI (include/ep.h): argument checks, the SM budget and
// kernel launches. No allocation, no synchronisation except ep_get_status.
//
// The SM budget follows DeepEP's Buffer.set_num_sms ("How DeepEP Utilizes TMA
// Instructions for Minimal SM Usage on Hopper GPUs", Minimal SM Occupancy
// Configuration): a process-wide setting read at every launch. Dispatch and
// combine launch at most that many CTAs, each requesting more than half of an
// SM's shared memory, so each CTA has an SM to itself and the grid occupies
// exactly that many SMs. The shared-memory request itself goes through the
// max-dynamic-shared-memory function attribute, as DeepEP's
// SET_SHARED_MEMORY_FOR_TMA does (same page, Dynamic Shared Memory
// Configuration).
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/ep.h"
#include "kernels.cuh"

namespace {

std::atomic<int> g_num_sms{0};
std::atomic<int> g_overlap_mode{0};  // 0 auto, 1 always, 2 never

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_smem_optin[kMaxDevices];

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// SM count and per-block shared-memory opt-in of the current device (cached).
bool device_limits(int* sm_count, int* smem_optin) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (dev >= 0 && dev < kMaxDevices) {
        int c = g_sm_count[dev].load(std::memory_order_relaxed);
        int s = g_smem_optin[dev].load(std::memory_order_relaxed);
        if (c > 0 && s > 0) {
            *sm_count = c;
            *smem_optin = s;
            return true;
        }
    }
    int c = 0, s = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&s, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return false;
    if (dev >= 0 && dev < kMaxDevices) {
        g_sm_count[dev].store(c, std::memory_order_relaxed);
        g_smem_optin[dev].store(s, std::memory_order_relaxed);
    }
    *sm_count = c;
    *smem_optin = s;
    return true;
}

int sms_in_effect(int sm_count) {
    const int b = g_num_sms.load(std::memory_order_relaxed);
    return (b <= 0 || b > sm_count) ? sm_count : b;
}

// SMs a copy kernel launched into `stream` uses: the budget, and no more
// than the SMs of the partition the stream belongs to, if any.
int sms_for_stream(int sm_count, cudaStream_t stream) {
    const int n = sms_in_effect(sm_count);
    const int part = ep::partition_sms(stream);
    return (part > 0 && part < n) ? part : n;
}

}  // namespace

namespace ep {

namespace {
thread_local int64_t t_call_bytes = 0;
}  // namespace

CallBytes::CallBytes(int64_t bytes) : saved_(t_call_bytes) { t_call_bytes = bytes; }
CallBytes::~CallBytes() { t_call_bytes = saved_; }

// Programmatic dependent launch (see launch_dependent): in the default mode
// while the SM budget covers the whole current device, or for a launch of a
// decode-size call into an SM-partition stream.
bool launch_overlap_allowed(cudaStream_t stream) {
    if (!EP_PDL) return false;
    const int mode = g_overlap_mode.load(std::memory_order_relaxed);
    if (mode == 1) return true;
    if (mode == 2) return false;
    if (partition_sms(stream) > 0) return t_call_bytes <= kPartitionOverlapBytes;
    int c = 0, s = 0;
    if (!device_limits(&c, &s)) return false;
    return sms_in_effect(c) == c;
}
}  // namespace ep

namespace {

ep_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

// Size limits, tested without forming a product that could overflow int64:
// T * K (token, expert) pairs and receive rows index with int32, and a row of
// H bf16 values is measured in uint32 bytes.
constexpr int64_t kMaxPairs = (int64_t{1} << 31) - 1;
bool pairs_fit(int64_t T, int K) { return T <= kMaxPairs / K; }
bool row_fits(int64_t H) { return H <= 0x7FFFFFF0 / 2; }

// Which combine kernel runs: the direct 16-byte gather (0), the bulk-copy
// staged ring (1), or the ring only at budgets of at most
// EP_COMBINE_TMA_MAX_SMS SMs (2). Both give identical results.
#ifndef EP_COMBINE_MODE
#define EP_COMBINE_MODE 0
#endif
#ifndef EP_COMBINE_TMA_MAX_SMS
#define EP_COMBINE_TMA_MAX_SMS 64
#endif

bool use_combine_tma(int K, int num_sms) {
    if (!ep::combine_tma_supported(K)) return false;
    if (EP_COMBINE_MODE == 1) return true;
    if (EP_COMBINE_MODE == 2) return num_sms <= EP_COMBINE_TMA_MAX_SMS;
    return false;
}

// Routing tables of at most this many entries are laid out by every CTA of
// the one-launch ep_layout_dispatch (a whole-table pass per CTA); larger ones
// take the layout kernel and dispatch as two launches.
constexpr int64_t kFusedMaxEntries = 4096;

#ifndef EP_LAYOUT_WIDE_CLUSTER
#define EP_LAYOUT_WIDE_CLUSTER 1
#endif

// Whether ep_layout_dispatch takes its two-launch form (the layout kernel,
// then dispatch) for a table of T*K entries on `s`, with the layout's plan:
// when the layout needs no workspace (one block, one 8-CTA cluster, or, for
// a table just past that, one 16-CTA cluster where the GPU can hold it) and
// either the table is too large for every CTA to histogram it cheaply, or
// launches may overlap on this stream (then the second launch costs
// nothing).
bool layout_dispatch_two_launches(int64_t T, int K, int E, cudaStream_t s, ep::LayoutPlan* lp) {
    *lp = ep::plan_layout(T * K, E);
    if (lp->workspace_bytes != 0) (void)ep::plan_layout_wide_cluster(T * K, E, lp);
    return lp->workspace_bytes == 0 && (T * K > kFusedMaxEntries || ep::launch_overlap_allowed(s));
}

// Host checks shared by ep_dispatch and ep_layout_dispatch.
ep_status_t check_dispatch(const uint16_t* x, int64_t T, int64_t H, int K, const int32_t* slot,
                           const float* topk_w, int64_t num_recv, const uint16_t* recv_x,
                           const float* recv_w, const int32_t* recv_src, const int32_t* status) {
    if (T < 0 || H <= 0 || H % 8 != 0 || K < 1 || K > EP_MAX_TOPK || num_recv < 0)
        return EP_ERR_INVALID;
    if (!pairs_fit(T, K) || num_recv > kMaxPairs || !row_fits(H)) return EP_ERR_UNSUPPORTED;
    if (T == 0) return EP_OK;
    if (x == nullptr || slot == nullptr || (num_recv > 0 && recv_x == nullptr)) return EP_ERR_INVALID;
    if (recv_w != nullptr && topk_w == nullptr) return EP_ERR_INVALID;
    if (!aligned(x, 16) || !aligned(recv_x, 16) || !aligned(slot, 4) || !aligned(topk_w, 4) ||
        !aligned(recv_w, 4) || !aligned(recv_src, 4) || !aligned(status, 4))
        return EP_ERR_INVALID;
    return EP_OK;
}

// (token, chunk) units the planner aims for per warp before it cuts rows finer.
#ifndef EP_DISPATCH_UNITS_PER_WARP
#define EP_DISPATCH_UNITS_PER_WARP 2
#endif

// Fills the kernel arguments: rows cut into equal 16-byte-multiple chunks
// that each fit one ring stage (after `reserve` bytes of other shared data).
// Small batches are cut finer (chunks of at least 512 bytes) until there are
// about two (token, chunk) units per warp of the grid, so a decode-size batch
// spreads over all its warps instead of leaving most of them idle.
ep_status_t plan_dispatch(ep::DispatchArgs* a, const uint16_t* x, int64_t T, int64_t H, int K,
                          const int32_t* slot, const float* topk_w, int64_t num_recv,
                          uint16_t* recv_x, float* recv_w, int32_t* recv_src, int32_t* status,
                          int smem_optin, size_t reserve, int num_sms, bool fused,
                          cudaStream_t stream) {
    a->x = reinterpret_cast<const uint8_t*>(x);
    a->T = T;
    a->row_bytes = static_cast<uint32_t>(H * 2);
    a->K = K;
    a->slot = slot;
    a->topk_w = topk_w;
    a->num_recv = num_recv;
    a->recv_x = reinterpret_cast<uint8_t*>(recv_x);
    a->recv_w = recv_w;
    a->recv_src = recv_src;
    a->status = status;
    a->ring_stages = ep::dispatch_ring_stages(fused, stream);
    uint32_t cap = ep::dispatch_stage_capacity(smem_optin, reserve, a->ring_stages);
    if (cap < 16) return EP_ERR_UNSUPPORTED;
#ifdef EP_DISPATCH_MAX_CHUNK
    if (cap > static_cast<uint32_t>(EP_DISPATCH_MAX_CHUNK)) cap = EP_DISPATCH_MAX_CHUNK;
#endif
    uint32_t n_chunks = (a->row_bytes + cap - 1) / cap;
    if (T > 0) {
        const int64_t target_units =
            static_cast<int64_t>(EP_DISPATCH_UNITS_PER_WARP) * num_sms * ep::dispatch_warps();
        const int64_t n_par = (target_units + T - 1) / T;
        const int64_t n_max = a->row_bytes / 512;  // chunks of at least 512 bytes
        const int64_t n_want = n_par < n_max ? n_par : n_max;
        if (n_want > n_chunks) n_chunks = static_cast<uint32_t>(n_want);
    }
#ifdef EP_DISPATCH_FORCE_CHUNKS
    if (static_cast<uint32_t>(EP_DISPATCH_FORCE_CHUNKS) > n_chunks) n_chunks = EP_DISPATCH_FORCE_CHUNKS;
#endif
    const uint32_t per = (a->row_bytes + n_chunks - 1) / n_chunks;
    a->chunk_bytes = (per + 15u) & ~15u;
    a->n_chunks = (a->row_bytes + a->chunk_bytes - 1) / a->chunk_bytes;
    a->stage_bytes = a->chunk_bytes;
    a->unit_base = 0;
    a->unit_count = T * static_cast<int64_t>(a->n_chunks);
    return EP_OK;
}

// Default percentage of a full-budget dispatch's units that go to the tail
// launch (DispatchArgs::tail_units; ep_set_dispatch_tail), for calls that
// move at least kTailMinBytes of receive rows with K >= 2. Back to back,
// dispatch alone and the step with combine after it: DeepSeek-V3 prefill
// (470 MB) 87.9 -> 76.8 and 171.6 -> 162.9 us, skewed Zipf 80.7 -> 70.1 and
// 152.0 -> 146.6 us, T=16384 (1.9 GB) 352 -> 314 us for dispatch. A fifth
// to two fifths measured within 1 us of each other. Smaller calls, mostly
// in L2, gain nothing; with K = 1 (as many bytes read as written) dispatch
// alone measured 2.5 us slower.
#ifndef EP_DISPATCH_TAIL_PERCENT
#define EP_DISPATCH_TAIL_PERCENT 30
#endif
constexpr int64_t kTailMinBytes = int64_t{192} << 20;
// Default percentage of a combine's units that go to a tail launch, under
// the same conditions as dispatch's (ep_set_combine_tail). Its SMs spread
// less than dispatch's, but a tail still helps: back to back, DeepSeek-V3
// prefill combine 78.9 -> 76.3 us, T=16384 316.5 -> 304.6 us; the steps
// with dispatch 162.1 -> 161.8, 635.5 -> 628.5 and skewed Zipf 147.4 ->
// 145.9 us (10 % and 20 % measured between none and this).
#ifndef EP_COMBINE_TAIL_PERCENT
#define EP_COMBINE_TAIL_PERCENT 30
#endif
std::atomic<int> g_combine_tail_percent{EP_COMBINE_TAIL_PERCENT};

// Tail share for this combine call (0: one persistent launch): as
// dispatch_tail_units, on the whole GPU with launches overlapping, for
// calls of at least kTailMinBytes of rows with K >= 2.
int combine_tail_percent(int64_t T, int64_t H, int K, int n, int sm_count, cudaStream_t s) {
    const int percent = g_combine_tail_percent.load(std::memory_order_relaxed);
    if (percent <= 0 || K < 2 || n < sm_count || !ep::launch_overlap_allowed(s)) return 0;
    return T * K * 2 * H >= kTailMinBytes ? percent : 0;
}
// Largest share of x a ring launch prefetches for its tail (a quarter of
// GB300's L2; DispatchArgs::tail_l2_prefetch).
constexpr int64_t kTailPrefetchMaxBytes = int64_t{32} << 20;
std::atomic<int> g_tail_percent{EP_DISPATCH_TAIL_PERCENT};

// Tail units for this call (0: one persistent launch): only on the whole
// GPU, where launches may overlap (the tail starts while the ring runs),
// and only while every ring warp keeps at least two units.
int64_t dispatch_tail_units(const ep::DispatchArgs& a, int n, int sm_count, cudaStream_t s) {
    const int percent = g_tail_percent.load(std::memory_order_relaxed);
    if (percent <= 0 || n < sm_count || !ep::launch_overlap_allowed(s)) return 0;
    if (a.K < 2 || a.T * a.K * static_cast<int64_t>(a.row_bytes) < kTailMinBytes) return 0;
    const int64_t tail = a.unit_count * percent / 100;
    const int64_t ring = a.unit_count - tail;
    return ring >= 2 * static_cast<int64_t>(n) * ep::dispatch_warps() ? tail : 0;
}

}  // namespace

extern "C" {

int ep_set_num_sms(int num_sms) {
    if (num_sms < 0) return -1;
    g_num_sms.store(num_sms, std::memory_order_relaxed);
    return num_sms;
}

int ep_get_num_sms(void) { return g_num_sms.load(std::memory_order_relaxed); }

int ep_set_launch_overlap(int mode) {
    if (mode < 0 || mode > 2) return -1;
    g_overlap_mode.store(mode, std::memory_order_relaxed);
    return mode;
}

int ep_get_launch_overlap(void) { return g_overlap_mode.load(std::memory_order_relaxed); }

int ep_set_dispatch_tail(int percent) {
    if (percent < 0 || percent > 90) return -1;
    g_tail_percent.store(percent, std::memory_order_relaxed);
    return percent;
}

int ep_get_dispatch_tail(void) { return g_tail_percent.load(std::memory_order_relaxed); }

int ep_set_combine_tail(int percent) {
    if (percent < 0 || percent > 90) return -1;
    g_combine_tail_percent.store(percent, std::memory_order_relaxed);
    return percent;
}

int ep_get_combine_tail(void) { return g_combine_tail_percent.load(std::memory_order_relaxed); }

int ep_combine_launches(int64_t T, int64_t H, int K, void* stream) {
    if (T < 0 || H <= 0 || H % 8 != 0 || K < 1 || K > EP_MAX_TOPK || !row_fits(H) ||
        !pairs_fit(T, K))
        return -1;
    if (T == 0) return 0;
    const ep::CallBytes call_bytes(T * K * 2 * H);
    int sm_count = 0, smem_optin = 0;
    if (!device_limits(&sm_count, &smem_optin)) return -1;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int n = sms_for_stream(sm_count, s);
    if (use_combine_tma(K, n)) return 1;
    return combine_tail_percent(T, H, K, n, sm_count, s) > 0 ? 2 : 1;
}

int ep_num_sms_in_effect(void) {
    int c = 0, s = 0;
    if (!device_limits(&c, &s)) return -1;
    return sms_in_effect(c);
}

size_t ep_layout_workspace_bytes(int64_t T, int K, int E) {
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS || !pairs_fit(T, K))
        return 0;
    return ep::plan_layout(T * K, E).workspace_bytes;
}

int ep_layout_launches(int64_t T, int K, int E) {
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS || !pairs_fit(T, K))
        return -1;
    const ep::LayoutPlan p = ep::plan_layout(T * K, E);
    if (p.num_tiles == 1 || p.cluster || p.coop) return 1;
    return p.num_tiles <= 512 ? 2 : 3;
}

int64_t ep_dispatch_chunk_bytes(int64_t T, int64_t H, int K) {
    if (T < 0 || H <= 0 || H % 8 != 0 || K < 1 || K > EP_MAX_TOPK || !row_fits(H) ||
        !pairs_fit(T, K))
        return -1;
    int sm_count = 0, smem_optin = 0;
    if (!device_limits(&sm_count, &smem_optin)) return -1;
    ep::DispatchArgs a{};
    if (plan_dispatch(&a, nullptr, T, H, K, nullptr, nullptr, 0, nullptr, nullptr, nullptr,
                      nullptr, smem_optin, 0, sms_in_effect(sm_count), false, nullptr) != EP_OK)
        return -1;
    return a.chunk_bytes;
}

int ep_dispatch_ring_stages(void) { return ep::dispatch_ring_stages(false, nullptr); }

int ep_layout_dispatch_launches(int64_t T, int64_t H, int K, int E, void* stream) {
    if (E < 1 || E > EP_MAX_EXPERTS) return -1;
    const int d = ep_dispatch_launches(T, H, K, stream);
    if (d <= 0) return d;
    const ep::CallBytes call_bytes(T * K * 2 * H);
    ep::LayoutPlan lp{};
    const bool two = layout_dispatch_two_launches(T, K, E, static_cast<cudaStream_t>(stream), &lp);
    return two ? 1 + d : 1;  // the two-launch form's layout is one launch
}

int ep_dispatch_launches(int64_t T, int64_t H, int K, void* stream) {
    if (T < 0 || H <= 0 || H % 8 != 0 || K < 1 || K > EP_MAX_TOPK || !row_fits(H) ||
        !pairs_fit(T, K))
        return -1;
    if (T == 0) return 0;
    const ep::CallBytes call_bytes(T * K * 2 * H);
    int sm_count = 0, smem_optin = 0;
    if (!device_limits(&sm_count, &smem_optin)) return -1;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int n = sms_for_stream(sm_count, s);
    ep::DispatchArgs a{};
    if (plan_dispatch(&a, nullptr, T, H, K, nullptr, nullptr, 0, nullptr, nullptr, nullptr,
                      nullptr, smem_optin, 0, n, false, s) != EP_OK)
        return -1;
    return dispatch_tail_units(a, n, sm_count, s) > 0 ? 2 : 1;
}

ep_status_t ep_get_dispatch_layout(const int64_t* topk_idx, int64_t T, int K, int E,
                                   int32_t* counts, int32_t* offsets, int32_t* slot,
                                   void* workspace, size_t workspace_bytes, int32_t* status,
                                   void* stream) {
    ep::ApiRange range("ep_get_dispatch_layout");
    if (T < 0 || K < 1 || K > EP_MAX_TOPK || E < 1) return EP_ERR_INVALID;
    if (E > EP_MAX_EXPERTS) return EP_ERR_UNSUPPORTED;
    if (!pairs_fit(T, K)) return EP_ERR_UNSUPPORTED;
    if (counts == nullptr || offsets == nullptr) return EP_ERR_INVALID;
    if (T > 0 && (topk_idx == nullptr || slot == nullptr)) return EP_ERR_INVALID;
    if (!aligned(topk_idx, 8) || !aligned(counts, 4) || !aligned(offsets, 4) || !aligned(slot, 4) ||
        !aligned(status, 4))
        return EP_ERR_INVALID;
    ep::LayoutPlan plan = ep::plan_layout(T * K, E);
    if (plan.workspace_bytes > 0) {
        if (workspace == nullptr || workspace_bytes < plan.workspace_bytes) return EP_ERR_WORKSPACE;
        if (!aligned(workspace, 16)) return EP_ERR_INVALID;
#if EP_LAYOUT_WIDE_CLUSTER
        // the workspace is asked for by size alone; a table that one 16-CTA
        // cluster can lay out leaves it unused where the GPU holds one
        (void)ep::plan_layout_wide_cluster(T * K, E, &plan);
#endif
    }
    return from_cuda(ep::launch_layout(topk_idx, T * K, E, counts, offsets, slot, workspace, plan,
                                       status, static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_dispatch(const uint16_t* x, int64_t T, int64_t H, int K, const int32_t* slot,
                        const float* topk_w, int64_t num_recv, uint16_t* recv_x, float* recv_w,
                        int32_t* recv_src, int32_t* status, void* stream) {
    ep::ApiRange range("ep_dispatch");
    ep_status_t st = check_dispatch(x, T, H, K, slot, topk_w, num_recv, recv_x, recv_w, recv_src,
                                    status);
    if (st != EP_OK || T == 0) return st;
    const ep::CallBytes call_bytes(T * K * 2 * H);
    int sm_count = 0, smem_optin = 0;
    if (!device_limits(&sm_count, &smem_optin)) return EP_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int n = sms_for_stream(sm_count, s);
    ep::DispatchArgs a{};
    st = plan_dispatch(&a, x, T, H, K, slot, topk_w, num_recv, recv_x, recv_w, recv_src, status,
                       smem_optin, 0, n, false, s);
    if (st != EP_OK) return st;
    // an early-started kernel brings its first rows into L2 while it waits
    a.l2_prefetch = (n >= sm_count && ep::launch_overlap_allowed(s)) ? 1 : 0;
    a.tail_units = dispatch_tail_units(a, n, sm_count, s);
    return from_cuda(ep::launch_dispatch(a, n, smem_optin, s));
}

ep_status_t ep_layout_dispatch(const int64_t* topk_idx, const uint16_t* x, int64_t T, int64_t H,
                               int K, int E, const float* topk_w, int64_t num_recv, int32_t* counts,
                               int32_t* offsets, int32_t* slot, uint16_t* recv_x, float* recv_w,
                               int32_t* recv_src, int32_t* status, void* stream) {
    ep::ApiRange range("ep_layout_dispatch");
    if (E < 1) return EP_ERR_INVALID;
    if (E > EP_MAX_EXPERTS) return EP_ERR_UNSUPPORTED;
    if (counts == nullptr || offsets == nullptr || !aligned(counts, 4) || !aligned(offsets, 4))
        return EP_ERR_INVALID;
    if (T > 0 && (topk_idx == nullptr || !aligned(topk_idx, 8))) return EP_ERR_INVALID;
    ep_status_t st = check_dispatch(x, T, H, K, slot, topk_w, num_recv, recv_x, recv_w, recv_src,
                                    status);
    if (st != EP_OK) return st;
    const ep::CallBytes call_bytes(T * K * 2 * H);
    int sm_count = 0, smem_optin = 0;
    if (!device_limits(&sm_count, &smem_optin)) return EP_ERR_CUDA;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int n = sms_for_stream(sm_count, s);
    // Two launches (the layout kernel, then dispatch) when the layout needs
    // no workspace and either the table is too large for every CTA to
    // histogram it cheaply, or launches may overlap on this stream (then the
    // second launch costs nothing). Dispatch's first row loads then overlap
    // the layout: its predecessor is that layout kernel, which does not
    // write x. Otherwise one launch does both.
    if (T > 0) {
        ep::LayoutPlan lp{};
        if (layout_dispatch_two_launches(T, K, E, s, &lp)) {
            cudaError_t e = ep::launch_layout(topk_idx, T * K, E, counts, offsets, slot, nullptr,
                                              lp, status, s);
            if (e != cudaSuccess) return EP_ERR_CUDA;
            ep::DispatchArgs a{};
            st = plan_dispatch(&a, x, T, H, K, slot, topk_w, num_recv, recv_x, recv_w, recv_src,
                               status, smem_optin, 0, n, false, s);
            if (st != EP_OK) return st;
            a.x_ready = 1;
            a.l2_prefetch = n >= sm_count ? 1 : 0;
            a.tail_units = dispatch_tail_units(a, n, sm_count, s);
            // the tail's x rows, when they fit a quarter of L2
            a.tail_l2_prefetch =
                (a.tail_units > 0 &&
                 a.tail_units * static_cast<int64_t>(a.chunk_bytes) <= kTailPrefetchMaxBytes)
                    ? 1
                    : 0;
            return from_cuda(ep::launch_dispatch(a, n, smem_optin, s));
        }
    }
    ep::DispatchArgs a{};
    // histograms, 16-byte alignment, the CTA's own keys and slots
    const size_t hist = 2 * sizeof(int32_t) * static_cast<size_t>(E) + 16 + ep::kFusedOwnBytes;
    st = plan_dispatch(&a, x, T, H, K, slot, topk_w, num_recv, recv_x, recv_w, recv_src, status,
                       smem_optin, hist, n, true, s);
    if (st != EP_OK) return st;
    ep::FusedLayoutArgs f{};
    f.idx = topk_idx;
    f.E = E;
    f.counts = counts;
    f.offsets = offsets;
    f.slot = slot;
    return from_cuda(ep::launch_layout_dispatch(a, f, n, s));
}

ep_status_t ep_combine(const uint16_t* expert_out, int64_t num_recv, const int32_t* slot,
                       const float* topk_w, int64_t T, int64_t H, int K, uint16_t* y,
                       int32_t* status, void* stream) {
    ep::ApiRange range("ep_combine");
    if (T < 0 || H <= 0 || H % 8 != 0 || K < 1 || K > EP_MAX_TOPK || num_recv < 0)
        return EP_ERR_INVALID;
    if (!pairs_fit(T, K) || num_recv > kMaxPairs || !row_fits(H)) return EP_ERR_UNSUPPORTED;
    if (T == 0) return EP_OK;
    if (slot == nullptr || topk_w == nullptr || y == nullptr ||
        (num_recv > 0 && expert_out == nullptr))
        return EP_ERR_INVALID;
    if (!aligned(expert_out, 16) || !aligned(y, 16) || !aligned(slot, 4) || !aligned(topk_w, 4) ||
        !aligned(status, 4))
        return EP_ERR_INVALID;
    const ep::CallBytes call_bytes(T * K * 2 * H);
    int sm_count = 0, smem_optin = 0;
    if (!device_limits(&sm_count, &smem_optin)) return EP_ERR_CUDA;
    ep::CombineArgs a{};
    a.expert_out = reinterpret_cast<const uint8_t*>(expert_out);
    a.num_recv = num_recv;
    a.slot = slot;
    a.topk_w = topk_w;
    a.T = T;
    a.row_bytes = static_cast<uint32_t>(H * 2);
    a.K = K;
    a.y = reinterpret_cast<uint8_t*>(y);
    a.status = status;
    const int n = sms_for_stream(sm_count, static_cast<cudaStream_t>(stream));
    a.tail_percent = combine_tail_percent(T, H, K, n, sm_count, static_cast<cudaStream_t>(stream));
    if (use_combine_tma(K, n))
        return from_cuda(ep::launch_combine_tma(a, n, smem_optin, static_cast<cudaStream_t>(stream)));
    return from_cuda(ep::launch_combine(a, n, static_cast<cudaStream_t>(stream)));
}

ep_status_t ep_get_status(const int32_t* status, void* stream) {
    if (status == nullptr) return EP_ERR_INVALID;
    int32_t v = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&v, status, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return EP_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return EP_ERR_CUDA;
    return static_cast<ep_status_t>(v);
}

const char* ep_status_string(ep_status_t s) {
    switch (s) {
        case EP_OK: return "ok";
        case EP_ERR_INVALID: return "invalid argument";
        case EP_ERR_UNSUPPORTED: return "size beyond the supported limits";
        case EP_ERR_CUDA: return "CUDA runtime error";
        case EP_ERR_TIMEOUT: return "bounded device wait gave up";
        case EP_ERR_BAD_EXPERT: return "expert id outside [0, E) and not -1";
        case EP_ERR_BAD_SLOT: return "slot beyond the receive buffer";
        case EP_ERR_WORKSPACE: return "layout workspace too small";
    }
    return "unknown status";
}

}  // extern "C"
