// kernels.cuh -- internal launch interface between the C ABI (ep_api.cu) and
// the kernels (layout.cu, dispatch.cu, combine.cu). Not part of the ABI.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

// NVTX ranges around the C ABI calls, so a profiler's timeline (Nsight
// Systems) attributes each launch to ep_get_dispatch_layout, ep_dispatch,
// ep_combine, ... The NVTX 3 header is self-contained; with no profiler
// attached a range costs a check of one function pointer. -DEP_NVTX=0
// compiles them out.
#ifndef EP_NVTX
#define EP_NVTX 1
#endif
#if EP_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace ep {

// Scoped NVTX range named after the entry point (a string literal).
struct ApiRange {
    explicit ApiRange(const char* name) {
#if EP_NVTX
        nvtxRangePushA(name);
#else
        (void)name;
#endif
    }
    ~ApiRange() {
#if EP_NVTX
        nvtxRangePop();
#endif
    }
    ApiRange(const ApiRange&) = delete;
    ApiRange& operator=(const ApiRange&) = delete;
};

// ---- layout ---------------------------------------------------------------

struct LayoutPlan {
    int warps;       // warps per block of the tile kernels
    int rounds;      // 32-entry rounds per warp per tile
    int64_t tile;    // entries per tile = warps * 32 * rounds
    int num_tiles;   // 1 => single fused launch, no workspace
    bool cluster;    // one thread-block cluster (no workspace)
    bool coop;       // one cooperative launch (else tile + finish launches)
    size_t smem;     // dynamic shared memory of the tile kernels
    size_t counts_off;       // workspace byte offset of tile_counts (num_tiles > 1)
    size_t workspace_bytes;  // 0 when num_tiles == 1
};

LayoutPlan plan_layout(int64_t N, int E);

// For tables that plan_layout gives a workspace but that fit one cluster of
// up to 16 CTAs (a non-portable cluster size) where the GPU can hold it: a
// plan for that cluster, with no workspace. For ep_layout_dispatch, which
// has none; ep_get_dispatch_layout keeps the plan that depends on the sizes
// alone (ep_layout_workspace_bytes). False where it does not apply.
bool plan_layout_wide_cluster(int64_t N, int E, LayoutPlan* out);

// `workspace` (16-byte aligned, plan.workspace_bytes) holds the barrier
// words and the [tiles][E] counts.
cudaError_t launch_layout(const int64_t* idx, int64_t N, int E, int32_t* counts,
                          int32_t* offsets, int32_t* slot, void* workspace,
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
    int ring_stages;       // ring stages the rows were planned for (host side)
    // 1: x was complete before this kernel's predecessor on the stream began
    // (that predecessor is this library's layout kernel, launched just
    // before by ep_layout_dispatch, which never writes x), so the first row
    // loads may go out before the kernel waits for its predecessor.
    int x_ready;
    // 1: while the first store still waits for the kernel before it (the
    // layout kernel, when launches overlap), bring the warp's next rows
    // into L2. Set at the full SM budget with launch overlap in effect,
    // where dispatch is bound by DRAM (DeepSeek-V3 step -3.2 us); on a
    // partial budget the SMs' own write path bounds it, and in the
    // one-launch form (tables that need a workspace, whose per-CTA layout
    // is long) the prefetched rows only crowd L2 (+1-2 %).
    int l2_prefetch;
    // This launch moves units [unit_base, unit_base + unit_count) of the
    // T * n_chunks (token, chunk) units.
    int64_t unit_base;
    int64_t unit_count;
    // Units the host gives to a tail launch (launch_dispatch), 0 for none.
    // At the full budget, with launches overlapping, the SMs do not move
    // bytes equally fast: under the same load some finish an equal share of
    // the units 25-35 % later than others (by SM, the same pattern launch
    // after launch). So the ring launch takes all but the last tail_units,
    // split evenly, and a second launch of many small CTAs (2 or 4 warps,
    // one unit each) takes the rest; those CTAs need more shared
    // memory than an SM has beside a ring CTA, so each starts only on an SM
    // whose ring CTA has finished, and the SMs that finish first take most
    // of the tail (the block scheduler serves as the work queue).
    int64_t tail_units;
    // 1: the ring launch, while the layout kernel of ep_layout_dispatch
    // holds back its first store, also brings the tail's rows of x into L2
    // (when they take at most a quarter of L2; larger ones are evicted
    // before the tail reads them). DeepSeek-V3 prefill step 162.4 ->
    // 161.0 us; T=3072 125.6 -> 123.2 us.
    int tail_l2_prefetch;
    // 1 in the tail launch: its CTAs start without waiting for the ring
    // launch (they only read what the ring launch read, which was complete
    // before the ring launch let them launch); its last CTA waits for the
    // ring launch to complete, so the tail launch completes after it.
    int tail;
};

// Routing inputs and layout outputs of the fused layout + dispatch kernel.
struct FusedLayoutArgs {
    const int64_t* idx;
    int E;
    int32_t* counts;
    int32_t* offsets;
    int32_t* slot;      // the same array as DispatchArgs::slot, written by the kernel
    uint32_t hist_off;  // shared-memory byte offset of its 2*E histogram words
    // Shared-memory byte offset of the CTA's own entries (kFusedOwnCap
    // int16 expert keys, then kFusedOwnCap int32 slots), or 0 when some CTA
    // has more entries than that (its slots then go through global memory).
    uint32_t own_off;
};
// Routing entries a fused-kernel CTA keeps in shared memory.
constexpr int kFusedOwnCap = 1024;
constexpr size_t kFusedOwnBytes = kFusedOwnCap * (sizeof(int16_t) + sizeof(int32_t));

cudaError_t launch_dispatch(const DispatchArgs& a, int num_sms, int smem_optin,
                            cudaStream_t stream);

// Layout and dispatch in one launch (every CTA computes the layout of its
// own tokens). a.slot must equal f.slot.
cudaError_t launch_layout_dispatch(const DispatchArgs& a, FusedLayoutArgs f, int num_sms,
                                   cudaStream_t stream);

// Largest ring stage (bytes, multiple of 16) dispatch can use on a device
// whose per-block shared-memory opt-in limit is `smem_optin`, after
// reserving `reserve` bytes for other shared data.
uint32_t dispatch_stage_capacity(int smem_optin, size_t reserve, int stages);
// Stages of the dispatch ring the next launch into `stream` will use
// (fused: the layout-plus-dispatch kernel); plan rows with the same number.
int dispatch_ring_stages(bool fused, cudaStream_t stream);

// Warps per dispatch CTA.
int dispatch_warps();

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
    // Percentage of the units a tail launch takes (0: one persistent
    // launch); set by the host where dispatch's tail applies, see
    // launch_shape in combine.cu.
    int tail_percent;
    // Set by launch_shape per launch: units [unit_base, unit_base +
    // unit_count) of the shape's T * column-block units, and 1 in the tail
    // launch (its CTAs skip the wait for the persistent launch but the last).
    int64_t unit_base;
    int64_t unit_count;
    int tail;
};

cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t stream);

// Combine with the expert rows staged through a per-warp bulk-copy ring
// (combine_tma.cu); K <= 8 only.
bool combine_tma_supported(int K);
cudaError_t launch_combine_tma(const CombineArgs& a, int num_sms, int smem_optin,
                               cudaStream_t stream);

// Launch a kernel of the hot path. With programmatic dependent launch the
// launch may start while the previous kernel on the stream finishes: its CTAs
// become resident and wait in griddep_wait(), which every such kernel calls
// before touching global memory, so the launch latency overlaps the previous
// kernel's tail. On the DeepSeek-V3 prefill step this saves ~2 us of ~180;
// on the decode step (T=128) 3-8 us of ~16-39.
// By default it is used only while the SM budget covers the whole GPU, or
// for decode-size calls into an SM-partition stream
// (launch_overlap_allowed). A smaller budget on an ordinary stream means
// the GPU is shared with concurrent work on SMs the hardware picks, and
// there an early-launched kernel may land on an SM the foreign work keeps
// busy: beside an ALU-bound kernel on the other SMs, the decode step on 24
// SMs took twice as long with early launches, and prefill dispatch +
// combine 3-6 % longer. A partition stream's kernels run only on the
// partition's SMs, where nothing foreign can sit.
#ifndef EP_PDL
#define EP_PDL 1
#endif
bool launch_overlap_allowed(cudaStream_t stream);

// SMs of the partition `stream` belongs to (ep_sm_partition), or 0 for any
// other stream.
int partition_sms(cudaStream_t stream);

// Row bytes the current C ABI call moves (0 for the layout), set for the
// call's duration by its entry point. Inside an SM partition, launches
// overlap only for calls that move at most kPartitionOverlapBytes
// (decode-size batches): there the early launches take the decode step on
// 24 SMs from ~30 to ~22 us, while a prefill-size call measured 3-5 %
// slower with them than without (the next kernel's CTAs then wait for the
// partition's own SMs to drain).
constexpr int64_t kPartitionOverlapBytes = int64_t{64} << 20;
class CallBytes {
  public:
    explicit CallBytes(int64_t bytes);
    ~CallBytes();
    CallBytes(const CallBytes&) = delete;
    CallBytes& operator=(const CallBytes&) = delete;

  private:
    int64_t saved_;
};

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), int grid, int block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(block));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = launch_overlap_allowed(stream) ? 1 : 0;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Dynamic shared memory that makes a CTA the only one resident on its SM
// (more than half of an SM's shared memory), so a grid of n CTAs occupies
// exactly n SMs.
constexpr size_t kExclusiveSmem = 120 * 1024;

}  // namespace ep
