// work_split.cuh -- how the copy kernels split their (token, chunk) units
// over warps, with 32-bit integer arithmetic whenever the sizes allow.
//
// A 64-bit integer division is a software routine of dozens of dependent
// instructions on the GPU; at decode sizes the few in each kernel's
// prologue cost a measurable part of a call of about ten microseconds.
// Every realistic size (fewer than 2^31 units, fewer than 2^16 warps) takes
// the 32-bit path; the results are identical either way.
#pragma once

#include <cstdint>

namespace ep {

// floor(x / d) for x >= 0, d > 0.
__device__ __forceinline__ int64_t div_floor(int64_t x, int64_t d) {
    if (x <= 0xFFFFFFFFll && d <= 0xFFFFFFFFll)
        return static_cast<uint32_t>(x) / static_cast<uint32_t>(d);
    return x / d;
}

// First unit of part g when `units` units are cut into W contiguous parts of
// near-equal size: floor(units * g / W), for 0 <= g <= W.
__device__ __forceinline__ int64_t split_begin(int64_t units, int64_t g, int64_t W) {
    if (units <= 0x7FFFFFFFll && W <= 0xFFFFll) {
        // units * g / W = q * g + (r * g) / W with q, r = units divmod W;
        // r * g < W^2 < 2^32
        const uint32_t w = static_cast<uint32_t>(W), gg = static_cast<uint32_t>(g);
        const uint32_t q = static_cast<uint32_t>(units) / w;
        const uint32_t r = static_cast<uint32_t>(units) - q * w;
        return static_cast<int64_t>(q) * gg + (r * gg) / w;
    }
    return units * g / W;
}

}  // namespace ep
