// combine_math.cuh -- the combine arithmetic, shared by the direct-gather
// combine (combine.cu) and the bulk-copy-staged one (combine_tma.cu), so both
// round exactly alike: bf16 widened to fp32 exactly (bit shift or mask), one
// fp32 fused multiply-add per k into an accumulator that starts at +0.0f,
// one bf16 round-to-nearest-even per output element.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace ep {

// acc[i] = fma(w, float(bf16 element i of v), acc[i]) for the 8 elements of v.
__device__ __forceinline__ void fma8(float (&acc)[8], float w, const uint4& v) {
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w, __uint_as_float(q[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
    }
}

// Same arithmetic as fma8 with packed fp32 pairs: acc2[i] holds elements
// 2i and 2i+1; fma.rn.f32x2 rounds each half exactly like fmaf.
__device__ __forceinline__ void fma8_x2(uint64_t (&acc2)[4], float w, const uint4& v) {
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
    uint64_t w2;
    asm("mov.b64 %0, {%1, %1};" : "=l"(w2) : "f"(w));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint64_t e2;
        asm("mov.b64 %0, {%1, %2};" : "=l"(e2) : "r"(q[i] << 16), "r"(q[i] & 0xFFFF0000u));
        asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc2[i]) : "l"(w2), "l"(e2));
    }
}

// Two fp32 values rounded to nearest-even bf16 and packed (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint4 round8(const float (&acc)[8]) {
    return make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                      pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
}

}  // namespace ep
