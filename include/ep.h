/*
 * ep.h -- C ABI of the GB300 (sm_103a) MoE token dispatch / combine library
 * (libep_gb300.so).
 *
 * Sources this interface follows (web pages; cited by title and section):
 *  [DeepEP-TMA]  "How DeepEP Utilizes TMA Instructions for Minimal SM Usage on
 *                Hopper GPUs" (instagit.com deep-dive on DeepSeek's DeepEP).
 *  [TMA-note]    TMA study note, mkbk-pku.cn (in Chinese): sections "Hopper
 *                architecture -- TMA" and "other TMA features".
 *  [TMA-atlas]   "tensor-memory-accelerator" (semiaifoundry.com atlas).
 *
 * What the library computes. DeepEP's dispatch takes a token matrix, a top-k
 * routing table and its weights ([DeepEP-TMA] "Practical Code Examples":
 * buffer.dispatch(hidden_states, topk_idx, topk_weights, num_experts)) and
 * copies every token row into a receive buffer of the expert it is routed to
 * ([DeepEP-TMA] "Asynchronous Copy Primitives", the receive loop). On one GPU
 * that is a pure HBM-to-HBM layout transform:
 *
 *   layout   counts[e]  = #{(t,k) : topk_idx[t,k] == e}
 *            offsets    = exclusive prefix of counts, offsets[E] = R
 *            slot[t,k]  = row of (t,k) in the receive buffer: experts in
 *                         ascending order, each expert's rows contiguous and
 *                         in ascending (t, k) order
 *   dispatch recv_x[slot[t,k], :] = x[t, :]              (bitwise copy)
 *   combine  y[t, :] = bf16_rne( sum over k = 0..K-1, in that order, as an
 *                      fp32 fused-multiply-add chain starting from +0.0f, of
 *                      topk_w[t,k] * float(expert_out[slot[t,k], :]) )
 *
 * The pages describe neither the layout call nor combine; the stable order,
 * the masking rule and the combine arithmetic above are this library's
 * readings (plainest reading of the MoE problem the pages state), chosen so
 * that every result has exactly one correct value.
 *
 * Conventions (all entry points):
 *  - Types. bf16 tensors are passed as uint16_t bit patterns (IEEE binary32
 *    upper half). Matrices are row-major and dense (row stride = width).
 *  - Memory. Every pointer except where noted is a DEVICE pointer on the
 *    current CUDA device. The caller allocates and owns every buffer,
 *    including the receive buffer and the layout workspace; the library
 *    allocates nothing and keeps no state besides the SM budget. (On one GPU
 *    this is what remains of DeepEP's pre-allocated communication Buffer.)
 *  - Streams. `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream). Every call only enqueues work and returns; ordering on
 *    the stream replaces the `event` DeepEP's dispatch returns.
 *  - Errors. Argument problems found on the host return at once, before any
 *    work is enqueued. Problems found on the device (an expert id out of
 *    range, a slot beyond the receive buffer, a bounded wait that gave up)
 *    skip the offending row and write their code into the optional device
 *    status word (first error wins); ep_get_status() reads it.
 *  - Alignment. x, recv_x, expert_out and y must be 16-byte aligned and H a
 *    multiple of 8 (rows are moved with 16-byte bulk copies, which need
 *    16-byte aligned addresses and sizes: [TMA-note] "Hopper architecture --
 *    TMA"). topk_idx must be 8-byte aligned; the int32/fp32 arrays 4-byte.
 *  - Masking. topk_idx[t,k] == -1 marks an unused entry: it gets slot -1 and
 *    every call skips it. Any other id outside [0, E) is skipped too and
 *    reported as EP_ERR_BAD_EXPERT.
 *  - Limits. 1 <= K <= 32, 1 <= E <= EP_MAX_EXPERTS, T*K < 2^31.
 *  - Threads. The SM budget is process-wide; concurrent calls from several
 *    host threads are the caller's to order.
 *  - First use. The first call that launches a given kernel shape (they
 *    differ by K, by the SM budget and by the table's size) loads that
 *    kernel into the CUDA context, and under CUDA's default lazy module
 *    loading that load waits until the device is idle: a call enqueued
 *    behind 100 ms of other work then returns after it. Warm each shape up
 *    before latency-critical work (or set CUDA_MODULE_LOADING=EAGER).
 *    Afterwards a call through the Python binding costs the host 6 us
 *    (ep_layout_dispatch 7-9 us; an empty torch kernel launch: 2 us).
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the shared library (built with hidden visibility by default). */
#if defined(__GNUC__)
#define EP_API __attribute__((visibility("default")))
#else
#define EP_API
#endif

#define EP_MAX_TOPK 32
#define EP_MAX_EXPERTS 4096

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID = 1,      /* bad argument (host): null, negative size, misalignment, K, H%8 */
    EP_ERR_UNSUPPORTED = 2,  /* sizes beyond the documented limits (host) */
    EP_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed (host) */
    EP_ERR_TIMEOUT = 4,      /* device: a bounded mbarrier wait gave up (~2 s) */
    EP_ERR_BAD_EXPERT = 5,   /* device: topk_idx outside [0, E) and not -1 */
    EP_ERR_BAD_SLOT = 6,     /* device: slot >= num_recv (receive buffer too small) */
    EP_ERR_WORKSPACE = 7     /* host: layout workspace smaller than required */
} ep_status_t;

/* SM budget, after DeepEP's Buffer.set_num_sms ([DeepEP-TMA] "Minimal SM
 * Occupancy Configuration"): dispatch and combine launch one CTA per SM on at
 * most this many SMs. 0 means all SMs. Values above the device's SM count
 * are clamped at launch. The layout is not budgeted (like the pages' budget,
 * this one covers the copy kernels): it runs a few microseconds on one
 * block, one 8-CTA cluster, or one block per tile of the routing table.
 * Returns the stored budget, or -1 (and changes nothing) if num_sms < 0. */
EP_API int ep_set_num_sms(int num_sms);

/* The stored SM budget (0 = all). */
EP_API int ep_get_num_sms(void);

/* Whether a kernel launch may overlap the tail of the previous kernel on the
 * stream (programmatic dependent launch; each kernel still waits for its
 * predecessor's results before touching global memory):
 *   0  auto (default): while the SM budget covers the whole GPU, and for
 *      calls into an SM-partition stream (ep_sm_partition) that move at
 *      most 64 MB of rows (decode-size batches; larger calls measured 3-5 %
 *      slower with overlapping launches there). A smaller budget on an
 *      ordinary stream usually means the GPU is shared with concurrent work,
 *      and there an early-launched kernel can land on an SM that work keeps
 *      busy (measured: the decode step on 24 SMs twice as long beside an
 *      ALU-bound kernel).
 *   1  always;  2  never.
 * Process-wide, like the SM budget. Returns the stored mode, or -1 (and
 * changes nothing) for any other value. */
EP_API int ep_set_launch_overlap(int mode);
EP_API int ep_get_launch_overlap(void);

/* Percentage (0 to 90, default 30) of a dispatch's (token, chunk) units
 * that go to its tail launch where it makes one (ep_dispatch_launches);
 * 0 keeps every dispatch to one persistent launch. Process-wide. Returns the
 * stored value, or -1 (and changes nothing) outside that range. */
EP_API int ep_set_dispatch_tail(int percent);
EP_API int ep_get_dispatch_tail(void);

/* The same for combine (0 to 90, default 30): under the same conditions as
 * dispatch's tail (ep_combine_launches), combine hands that share of its
 * (token, column block) units to a second launch of small CTAs. Returns the
 * stored value, or -1 (and changes nothing) outside that range. */
EP_API int ep_set_combine_tail(int percent);
EP_API int ep_get_combine_tail(void);

/* The number of SMs dispatch/combine will use on the current device: the
 * budget clamped to [1, SM count]. Returns -1 if the device can't be queried. */
EP_API int ep_num_sms_in_effect(void);

/* Bytes of device workspace ep_get_dispatch_layout needs for these sizes
 * (0 when none; then `workspace` may be NULL). Depends on sizes only. */
EP_API size_t ep_layout_workspace_bytes(int64_t T, int K, int E);

/* Kernel launches one ep_get_dispatch_layout call makes for these sizes on a
 * GPU where all of its tiles can be resident at once (1 for tables of up to
 * 128 tiles; 2 or 3 above that), for accounting in measurements; -1 for
 * invalid sizes. */
EP_API int ep_layout_launches(int64_t T, int K, int E);

/* Bytes per row chunk that ep_dispatch would use for these sizes at the
 * current SM budget on the current device: each bf16 row of 2*H bytes is cut
 * into equal 16-byte-multiple chunks, each one bulk load and K bulk stores
 * (one ring unit). For measurements that model the ring; -1 for invalid
 * sizes or when the device cannot be queried. */
EP_API int64_t ep_dispatch_chunk_bytes(int64_t T, int64_t H, int K);

/* Stages of the per-warp shared-memory ring ep_dispatch uses at the current
 * SM budget and launch-overlap mode: 3 while launches overlap (a dispatch CTA
 * then needs less shared memory, so its SM keeps a larger L1 share; measured
 * faster with the kernels overlapping), else 4. For measurements that model
 * the ring. */
EP_API int ep_dispatch_ring_stages(void);

/* Kernel launches one ep_dispatch call makes for these sizes on `stream`
 * (NULL: the legacy default stream) at the current SM budget and
 * launch-overlap mode: 2 when it splits the rows between a persistent launch
 * and a tail launch, else 1; the dispatch part of ep_layout_dispatch in its
 * two-launch form does the same. The split is made on the whole GPU, while
 * launches overlap, for calls of at least 192 MB of receive rows and K >= 2
 * (and a tail percentage above 0, ep_set_dispatch_tail). There, under one
 * load, some SMs move an equal share 25-35 % later than others (the same SMs
 * launch after launch), so the persistent launch takes 70 % of the (token,
 * chunk) units, split evenly, and the tail launch's
 * small CTAs take the rest, each starting only on an SM whose persistent CTA
 * has finished: the SMs that finish first take most of the tail. For
 * accounting in measurements; -1 for invalid sizes or when the device
 * cannot be queried. */
EP_API int ep_dispatch_launches(int64_t T, int64_t H, int K, void* stream);

/* Kernel launches one ep_layout_dispatch call makes for these sizes on
 * `stream` at the current SM budget and launch-overlap mode: 1 in its
 * one-launch form, else 1 for the layout plus ep_dispatch_launches. -1 for
 * invalid sizes or when the device cannot be queried. */
EP_API int ep_layout_dispatch_launches(int64_t T, int64_t H, int K, int E, void* stream);

/* Kernel launches one ep_combine call makes for these sizes on `stream` at
 * the current SM budget and launch-overlap mode: 2 where it hands part of
 * its units to a tail launch (the whole GPU, launches overlapping, at least
 * 192 MB of rows, K >= 2, a combine tail share above 0), else 1. -1 for
 * invalid sizes or when the device cannot be queried. */
EP_API int ep_combine_launches(int64_t T, int64_t H, int K, void* stream);

/* Layout (per-expert histogram, exclusive prefix sums and per-(token,k)
 * destination slot).
 *   topk_idx   int64 [T][K]   routing table (DeepEP's topk_idx)
 *   counts     int32 [E]      out: rows per expert
 *   offsets    int32 [E+1]    out: first row of each expert; offsets[E] = R
 *   slot       int32 [T][K]   out: receive row of (t,k), -1 if skipped
 *   workspace  device scratch of ep_layout_workspace_bytes(T,K,E) bytes,
 *              16-byte aligned. It carries two small words (owner tag and
 *              generation) from one call to the next for the kernels' grid
 *              barrier; any initial content is valid, so it never needs
 *              clearing, and within a process the barrier's targets never
 *              repeat. Calls that share a workspace must not overlap on the
 *              GPU. Tables that one 16-CTA thread-block cluster can lay out
 *              (up to 131,072 entries at E <= 256) leave it unused where the
 *              GPU can hold such a cluster; its size still depends on the
 *              sizes alone.
 *   status     int32 device word, nullable (device errors: BAD_EXPERT)
 * T == 0 is valid (counts and offsets are zeroed). */
EP_API ep_status_t ep_get_dispatch_layout(const int64_t* topk_idx, int64_t T, int K, int E,
                                   int32_t* counts, int32_t* offsets, int32_t* slot,
                                   void* workspace, size_t workspace_bytes,
                                   int32_t* status, void* stream);

/* Dispatch ([DeepEP-TMA] "Asynchronous Copy Primitives"): each warp's elected
 * lane bulk-copies token-row chunks global -> shared (completion on an
 * mbarrier) and shared -> global, once into shared memory and K times out.
 *   x          bf16 [T][H]
 *   slot       int32 [T][K]  from ep_get_dispatch_layout
 *   topk_w     fp32 [T][K]   nullable; needed only for recv_w
 *   num_recv   rows of recv_x (>= R = offsets[E]); larger slots -> BAD_SLOT
 *   recv_x     bf16 [num_recv][H] out
 *   recv_w     fp32 [num_recv] out, nullable: recv_w[slot[t,k]] = topk_w[t,k]
 *   recv_src   int32 [num_recv] out, nullable: recv_src[slot[t,k]] = t*K + k
 * Rows of recv_x no (t,k) maps to are left untouched. One persistent CTA per
 * SM of the budget, the (token, chunk) units split evenly over its warps;
 * on the whole GPU, with launches overlapping, calls of at least 192 MB of
 * receive rows (K >= 2) hand the last 30 % of the units to a second launch
 * of small CTAs (ep_dispatch_launches). */
EP_API ep_status_t ep_dispatch(const uint16_t* x, int64_t T, int64_t H, int K,
                        const int32_t* slot, const float* topk_w, int64_t num_recv,
                        uint16_t* recv_x, float* recv_w, int32_t* recv_src,
                        int32_t* status, void* stream);

/* Layout and dispatch in one call: the results of ep_get_dispatch_layout
 * (counts, offsets, slot) and of ep_dispatch (recv_x, recv_w, recv_src),
 * identical to calling the two in turn, with no workspace argument.
 *  - Small tables (at most 4096 entries) on a stream where launches may not
 *    overlap (a partial SM budget on an ordinary stream): one launch in
 *    which every CTA reads the whole routing table and lays out its own
 *    tokens (on GB300, T=128 top-8 on 24 SMs: a layout + dispatch + combine
 *    step takes 29.4 us with it, 33.4 us with the separate calls).
 *  - Otherwise, when the layout needs no workspace (one block or one
 *    thread-block cluster: at most 65,536 entries at E <= 256, or 131,072
 *    with a 16-CTA cluster where the GPU can hold one): the layout kernel
 *    and the dispatch kernel, with dispatch's first row loads (its whole
 *    ring; at the full SM budget also the next rows, into L2) issued while
 *    the layout runs (safe because this call launched that layout kernel
 *    itself, which never writes x): on GB300 the DeepSeek-V3 prefill step
 *    (T=4096 top-8, H=7168) takes 0.161-0.163 ms with it and 0.165 ms with
 *    the separate calls; T=16384 (131,072 entries, the 16-CTA cluster)
 *    0.635 vs 0.645 ms.
 *  - Larger tables fall back to the one-launch form, whose cost grows with
 *    T*K per CTA; call the two functions separately for those
 *    (ep_layout_dispatch_launches tells the forms apart).
 * Arguments as in those two calls; T == 0 still writes zero counts and
 * offsets. */
EP_API ep_status_t ep_layout_dispatch(const int64_t* topk_idx, const uint16_t* x, int64_t T,
                                      int64_t H, int K, int E, const float* topk_w,
                                      int64_t num_recv, int32_t* counts, int32_t* offsets,
                                      int32_t* slot, uint16_t* recv_x, float* recv_w,
                                      int32_t* recv_src, int32_t* status, void* stream);

/* Combine: weighted gather of the K expert rows of every token back into
 * token order (arithmetic in the header comment above).
 *   expert_out bf16 [num_recv][H]  rows in receive order
 *   slot       int32 [T][K]
 *   topk_w     fp32 [T][K]         routing weights in token order
 *   y          bf16 [T][H] out
 * A token whose K entries are all skipped gets +0.0. One persistent CTA per
 * SM of the budget, the (token, column block) units split evenly over its
 * warps; where dispatch would make a tail launch, combine hands the last
 * 30 % of its units to one too (ep_combine_launches). */
EP_API ep_status_t ep_combine(const uint16_t* expert_out, int64_t num_recv,
                       const int32_t* slot, const float* topk_w,
                       int64_t T, int64_t H, int K,
                       uint16_t* y, int32_t* status, void* stream);

/* Layout without a workspace argument, for callers that cannot allocate
 * device memory. The pages have no counterpart; this is a library addition.
 * Such callers include a serving engine that reserved nearly all of HBM up
 * front for weights and KV cache (an extra cudaMalloc would fail or fragment
 * its pool) and latency-critical pipelines (cudaMalloc/cudaFree may
 * synchronise the whole device). Same arguments and results as
 * ep_get_dispatch_layout, but the layout's scratch lives in a static device
 * array of EP_NOALLOC_SCRATCH_BYTES that every GPU loading the library keeps
 * until the process exits; this call allocates nothing.
 *  - Limit: sizes whose ep_layout_workspace_bytes(T,K,E) exceeds
 *    EP_NOALLOC_SCRATCH_BYTES are rejected with EP_ERR_UNSUPPORTED.
 *  - Set-up: the first call on each device (with that device current) looks
 *    up the array's device address and caches it with the id of the current
 *    CUDA context; make that first call before any stream capture. A
 *    cudaDeviceReset destroys the context and the array with it: the next
 *    call on that device (again outside any capture) looks the address up
 *    anew, and the array's contents start over.
 *  - Sharing: all calls share the array. Calls that overlap on the GPU (other
 *    streams or host threads) race on it; order them. Tables that one
 *    16-CTA thread-block cluster lays out (up to 131,072 entries at
 *    E <= 256, where the GPU holds such a cluster) do not use it. Nothing in it needs to
 *    start at zero: each call rewrites the counts it reads, and the one word
 *    it carries between calls is valid from any starting value. */
#define EP_NOALLOC_SCRATCH_BYTES (1u << 20)
EP_API ep_status_t ep_get_dispatch_layout_noalloc(const int64_t* topk_idx, int64_t T, int K, int E,
                                                  int32_t* counts, int32_t* offsets, int32_t* slot,
                                                  int32_t* status, void* stream);

/* SM partition: a stream whose kernels the hardware runs on a fixed set of
 * at least num_sms SMs, and a stream for the device's other SMs (CUDA green
 * contexts). The pages' SM budget ([DeepEP-TMA] "Minimal SM Occupancy
 * Configuration": a few SMs for communication, the rest for computation)
 * limits how many CTAs a kernel launches, not which SMs run them; a
 * partition fixes those SMs too.
 *   num_sms     SMs wanted (>= 1); rounded up to the device's partition
 *               granularity (8 SMs on GB300)
 *   stream      out: cudaStream_t (as void*) of the partition
 *   rest_stream out, nullable: cudaStream_t of the remaining SMs (NULL if
 *               none remain), for the work that runs beside the movement
 *   sms, rest_sms  out, nullable: SMs of each
 * On the current device. Calls with the same num_sms on the same device
 * return the same streams; partitions live until the process exits (the
 * caller must not destroy the streams). Every call of this library into the
 * partition stream uses at most its SMs (the budget still applies below
 * that), and under the default launch-overlap policy (mode 0) the launches
 * of decode-size calls may overlap the previous kernel's tail, since
 * nothing foreign can share those SMs (T=128 top-8, H=7168 on 24 SMs: 22 us
 * per step against 30 us on an ordinary stream).
 * Returns EP_ERR_UNSUPPORTED where the driver offers no green contexts or
 * num_sms exceeds the SM count; EP_ERR_INVALID for num_sms < 1 or a null
 * `stream`. The pages have no counterpart for the partition itself. */
EP_API ep_status_t ep_sm_partition(int num_sms, void** stream, void** rest_stream, int* sms,
                                   int* rest_sms);

/* Self-test of the failure path: launches one warp that waits, for at most
 * `limit_ns` nanoseconds (1 .. 2e9), on an mbarrier nothing completes, so the
 * bounded wait gives up and writes EP_ERR_TIMEOUT to *status (the way every
 * wait in the kernels ends if a copy never arrives). Like the copy kernels
 * after a timeout, it then waits once more, with the same bound, on each stage
 * of its three-stage ring that could still have a load in flight, and returns
 * after about four limits. For tests; it changes nothing else. */
EP_API ep_status_t ep_selftest_wait_timeout(int32_t* status, uint64_t limit_ns, void* stream);

/* Synchronises `stream`, then returns the device status word (an
 * ep_status_t), or EP_ERR_CUDA if the copy fails. Does not reset it. */
EP_API ep_status_t ep_get_status(const int32_t* status, void* stream);

/* Static description of a status code. */
EP_API const char* ep_status_string(ep_status_t s);

#ifdef __cplusplus
}
#endif
#endif /* EP_GB300_H */
