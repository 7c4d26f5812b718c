// routing.cuh -- device helpers shared by the layout kernels and the fused
// layout + dispatch kernel: expert ids, warp peer groups, block scan.
#pragma once

#include <cstdint>

namespace ep {

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
__device__ inline int64_t block_exclusive_scan(int64_t v, int64_t* total) {
    __shared__ int64_t warp_base[32];
    __shared__ int64_t block_total;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    int64_t incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int64_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) warp_base[warp] = incl;  // warp sum
    __syncthreads();
    if (warp == 0) {
        const int64_t s = lane < nwarps ? warp_base[lane] : 0;
        int64_t si = s;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int64_t o = __shfl_up_sync(0xFFFFFFFFu, si, d);
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

// Lanes of the warp whose key equals this lane's key (all invalid lanes,
// key -1, form one group). Built from one ballot per key bit: a handful of
// single-cycle votes instead of a warp match.
__device__ __forceinline__ uint32_t peers_of(int key, int key_bits) {
    const uint32_t valid = __ballot_sync(0xFFFFFFFFu, key >= 0);
    uint32_t m = key >= 0 ? valid : ~valid;
    for (int b = 0; b < key_bits; ++b) {
        const bool bit = (key >> b) & 1;
        const uint32_t ones = __ballot_sync(0xFFFFFFFFu, bit);
        m &= bit ? ones : ~ones;
    }
    return m;
}

// Bits needed for expert ids 0..E-1.
__device__ __forceinline__ int key_bits_for(int E) { return E > 1 ? 32 - __clz(E - 1) : 0; }

}  // namespace ep
