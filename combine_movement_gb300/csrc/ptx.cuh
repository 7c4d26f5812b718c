// ptx.cuh -- inline-PTX primitives for the bulk-copy (TMA) data path on
// sm_103a: single-lane election, mbarriers with bounded waits, and 1-D
// cp.async.bulk copies global<->shared. Written from the public PTX ISA.
//
// What each wraps, and where the pages use it:
//  * elect_one()          -- elect.sync; one lane per warp issues every bulk
//    copy ("How DeepEP Utilizes TMA Instructions for Minimal SM Usage on
//    Hopper GPUs", FAQ "Why does DeepEP use only one lane per warp").
//  * bulk_load / bulk_store / bulk_commit / bulk_wait_read -- DeepEP's
//    tma_load_1d / tma_store_1d / tma_store_wait (same page, "Asynchronous
//    Copy Primitives").
//  * mbar_* -- the completion barrier the copy engine updates when the bytes
//    have landed (TMA study note, mkbk-pku.cn, "Hopper architecture -- TMA",
//    workflow: init barrier, issue copy bound to it, hardware updates it,
//    consumer waits). Every wait here is bounded in time.
#pragma once

#include <cstdint>

namespace ep {

// Upper bound on any single mbarrier wait. A correct pipeline waits
// microseconds; after this long the kernel records EP_ERR_TIMEOUT and
// returns instead of spinning forever.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// True in exactly one lane of a fully converged warp.
__device__ __forceinline__ bool elect_one() {
    uint32_t is_elected;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(is_elected));
    return is_elected != 0;
}

// ---- mbarrier -----------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t arrivals) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(arrivals) : "memory");
}

// Make mbarrier initialisation (a generic-proxy write) visible to the async
// proxy, which completes transactions on it.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive once and add `bytes` to the transaction count the current phase
// must see before it completes.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

// Wait for the phase of parity `parity` to complete; false if it did not
// within `limit_ns` (kWaitLimitNs unless a self-test asks for less).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// After a ring wait gave up: wait again, each with the same bound, for the
// loads of ring units `first` .. `last` that may still be in flight (unit i
// lands in stage i % NS and completes phase (i / NS) & 1 of its barrier), so
// no bulk copy writes shared memory after the CTA has exited. Returns whether
// all of them arrived.
template <int NS>
__device__ __forceinline__ bool mbar_drain_bounded(uint32_t bar0, int64_t first, int64_t last,
                                                   uint64_t limit_ns = kWaitLimitNs) {
    bool all = true;
    for (int64_t i = first; i <= last; ++i)
        all &= mbar_wait_bounded(bar0 + 8u * static_cast<uint32_t>(i % NS),
                                 static_cast<uint32_t>((i / NS) & 1), limit_ns);
    return all;
}

// ---- L2 cache policies ---------------------------------------------------

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- 1-D bulk copies (no tensor map) -------------------------------------
// Sizes are multiples of 16 bytes; both addresses 16-byte aligned.

// global -> shared::cta; completes `bytes` transactions on mbarrier `bar`.
// (The shared::cluster destination form with a CTA-local address; no
// multicast.)
__device__ __forceinline__ void bulk_load(uint32_t dst_smem, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst_smem),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// shared::cta -> global, tracked by this thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void* dst, uint32_t src_smem, uint32_t bytes,
                                           uint64_t policy) {
    asm volatile(
        "cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst),
        "r"(src_smem), "r"(bytes), "l"(policy)
        : "memory");
}

// Bring `bytes` of global memory into L2 (no shared memory, no completion
// to wait for); a hint only.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes, uint64_t policy) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src),
                 "r"(bytes), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until at most N of this thread's bulk groups are incomplete.
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// ---- plain vector loads/stores for the combine path -----------------------

// 16-byte read-only load that does not allocate in L1 (each expert row is
// read exactly once).
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// The same load without `volatile`, so the compiler may schedule it freely
// among other loads. Only for addresses computed from data loaded after
// griddep_wait() (a combine row address comes from its slot), which keeps it
// behind that wait.
__device__ __forceinline__ uint4 ld_nc_v4_dep(const void* p) {
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

__device__ __forceinline__ void st_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// ---- programmatic dependent launch ------------------------------------------
// A kernel launched with programmatic stream serialization may start while
// the previous kernel on the stream is still running; griddep_wait() blocks
// until that kernel has completed and its memory is visible, so it must come
// before the first global-memory access. griddep_launch_dependents() lets the
// next such kernel begin launching now. Both are no-ops for ordinary launches.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Record the first device-side error (0 = none so far).
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
    if (status != nullptr) atomicCAS(status, 0, code);
}

}  // namespace ep
