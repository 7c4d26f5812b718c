// combine.cu -- gather every token's K expert rows back into token order and
// reduce them with the routing weights.
//
// The pages describe only DeepEP's dispatch ("How DeepEP Utilizes TMA
// Instructions for Minimal SM Usage on Hopper GPUs"); combine is its inverse
// in the MoE layer the page is about: y[t] = sum_k w[t,k] * expert_out[slot[t,k]].
// The arithmetic is fixed so the result is unique: fp32 accumulator starting
// at +0.0f, one fused multiply-add per k in ascending k (entries with slot < 0
// skipped), one bf16 round-to-nearest-even per output element.
//
// Mapping: persistent grid of one CTA per SM (the SM budget). A unit is one,
// two or four 512-byte column blocks of one token row (a block is 32 lanes x
// 16 bytes); every warp takes a contiguous, equal range of units, so the
// load is balanced to within one unit whatever T and the budget. For each
// token the warp reads slot and weight once (lanes k < K) and broadcasts
// them with warp shuffles; each lane then issues K independent 16-byte loads
// per column block of the unit (read-only path, no L1 allocation), widens
// bf16 to fp32 exactly (bit shift), runs the fma chain in k order and writes
// 16 bytes per block, so every warp store is a coalesced 512-byte row
// segment. Units whose K slots are all valid and which lie wholly inside the
// row take an unpredicated body whose fmas go in packed fp32 pairs
// (fma.rn.f32x2, the same rounding per element), for every K <= 8.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/ep.h"
#include "combine_math.cuh"
#include "kernels.cuh"
#include "ptx.cuh"
#include "work_split.cuh"

namespace ep {
namespace {

// Compiled shape per K: threads per CTA, 512-byte column blocks per unit,
// and whether expert rows are addressed by 32-bit slot index (one more
// multiply-add per load, fewer registers) instead of a 64-bit pointer per
// k. A lane issues all K x blocks loads of a unit before its fmas, and on a
// small SM budget each SM's read rate follows the bytes it keeps in flight,
// so each lane takes two (K = 1: four) blocks per unit with as many threads
// as the registers then hold without spilling. Each entry was the fastest
// measured at 16-48 SMs (thread counts that split evenly over the SM's four
// schedulers), and at 96 and 152 SMs, where HBM bounds K >= 4, it is as
// fast as or faster than 384 threads x 2 blocks.
struct CombineShape {
    int threads;
    int unroll;
    bool slot_rows;
};
constexpr CombineShape combine_shape(int KT) {
#ifdef EP_COMBINE_SHAPE_OVERRIDE
    // measurement builds: threads * 10 + column blocks, rows by slot index,
    // for every K <= 8
    if (KT > 0) return {EP_COMBINE_SHAPE_OVERRIDE / 10, EP_COMBINE_SHAPE_OVERRIDE % 10, true};
#endif
    switch (KT) {
        case 1: return {1024, 4, true};
        case 2: return {1024, 2, false};
        case 3: return {1024, 2, false};
        case 4: return {896, 2, true};
        case 5: return {640, 2, true};
        case 6: return {640, 2, true};
        case 7: return {512, 2, true};
        case 8: return {512, 2, true};
        default: return {768, 1, false};  // generic path, K > 8, below kGenericWideSms
    }
}
// The generic path (K > 8) runs 384 threads x 2 blocks from this many SMs up.
constexpr int kGenericWideSms = 96;
// A batch too small to give every budgeted SM one CTA of its K's shape (a
// decode step at a large budget) runs 384 threads x 2 blocks instead: 12
// warps per CTA spread it over more SMs.
constexpr int kSmallThreads = 384;
constexpr int kSmallUnroll = 2;

#ifndef EP_COMBINE_TAIL_WARPS
#define EP_COMBINE_TAIL_WARPS 4
#endif
#ifndef EP_COMBINE_TAIL_UNITS
#define EP_COMBINE_TAIL_UNITS 2
#endif

constexpr unsigned kFullMask = 0xFFFFFFFFu;
constexpr uint32_t kColBytes = 512;  // row bytes one warp covers per column block
constexpr int kGenericBatch = 8;     // k entries per batch of loads in the generic path

// KT > 0: K == KT known at compile time (slots, row pointers and weights in
// registers). KT == 0: any K <= 32, broadcast per unit. A unit is UN
// consecutive 512-byte column blocks of one token, so each lane keeps
// UN * K independent 16-byte loads in flight.
template <int KT, int kThreads, int kUnroll, bool kFast, bool kSlotRows>
__global__ void __launch_bounds__(kThreads, 1) combine_kernel(const CombineArgs a) {
    if (!a.tail || blockIdx.x == gridDim.x - 1) griddep_wait();
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    constexpr uint32_t kUnitBytes = kColBytes * kUnroll;
    const int64_t n_cb = (a.row_bytes + kUnitBytes - 1) / kUnitBytes;
    // this launch's units, split evenly over its warps
    const int64_t units = a.unit_count;
    const int64_t gw = static_cast<int64_t>(blockIdx.x) * nwarps + warp;
    const int64_t nw_total = static_cast<int64_t>(gridDim.x) * nwarps;
    const int64_t u0 = a.unit_base + split_begin(units, gw, nw_total);
    const int64_t u1 = a.unit_base + split_begin(units, gw + 1, nw_total);
    const int K = KT > 0 ? KT : a.K;
    constexpr int KR = KT > 0 ? KT : 1;

    int64_t tok = -1;
    // expert row of each k (row 0 where masked): a slot index or a pointer
    int32_t rowi[KR] = {};
    const uint8_t* rowp[KR] = {};
    auto row = [&](int k) -> const uint8_t* {
        return kSlotRows ? a.expert_out + static_cast<int64_t>(rowi[k]) * a.row_bytes : rowp[k];
    };
    float wk[KR];
    bool on[KR];
    bool all_on = false;  // every one of the token's K slots is valid (warp-uniform)
    int32_t s_lane = -1;
    float w_lane = 0.0f;

    // (token, column block) of the current unit, advanced without divisions
    int64_t t = div_floor(u0, n_cb);
    uint32_t cb = static_cast<uint32_t>(u0 - t * n_cb);
    for (int64_t u = u0; u < u1; ++u) {
        const uint32_t col0 = cb * kUnitBytes + lane * 16u;
        if (t != tok) {
            tok = t;
            int32_t s = lane < K ? __ldg(a.slot + t * K + lane) : -1;
            const float w = lane < K ? __ldg(a.topk_w + t * K + lane) : 0.0f;
            if (s >= a.num_recv) {
                set_status(a.status, EP_ERR_BAD_SLOT);
                s = -1;
            }
            s_lane = s;
            w_lane = w;
            if (KT > 0) {
#pragma unroll
                for (int k = 0; k < KR; ++k) {
                    const int32_t sk = __shfl_sync(kFullMask, s, k);
                    wk[k] = __shfl_sync(kFullMask, w, k);
                    on[k] = sk >= 0;
                    if (kSlotRows)
                        rowi[k] = sk < 0 ? 0 : sk;
                    else
                        rowp[k] = a.expert_out + static_cast<int64_t>(sk < 0 ? 0 : sk) * a.row_bytes;
                }
                all_on = __all_sync(kFullMask, lane >= K || s >= 0);
            }
        }
        // kFast, common case: no masked slot and the whole unit inside the
        // row, so loads and fmas need no per-element predicates, and the fmas
        // go in packed pairs.
        if (kFast && KT > 0 && all_on && (cb + 1) * kUnitBytes <= a.row_bytes) {
            uint4 v[kUnroll][KR];
#pragma unroll
            for (int k = 0; k < KR; ++k)
#pragma unroll
                for (int j = 0; j < kUnroll; ++j) v[j][k] = ld_nc_v4_dep(row(k) + col0 + j * kColBytes);
            float acc[kUnroll][8];
#pragma unroll
            for (int j = 0; j < kUnroll; ++j) {
                uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};  // +0.0f pairs
#pragma unroll
                for (int k = 0; k < KR; ++k) fma8_x2(acc2, wk[k], v[j][k]);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    asm("mov.b64 {%0, %1}, %2;"
                        : "=f"(acc[j][2 * i]), "=f"(acc[j][2 * i + 1])
                        : "l"(acc2[i]));
            }
            uint8_t* yrow = a.y + t * static_cast<int64_t>(a.row_bytes);
#pragma unroll
            for (int j = 0; j < kUnroll; ++j) st_v4(yrow + col0 + j * kColBytes, round8(acc[j]));
            if (++cb == n_cb) {
                cb = 0;
                ++t;
            }
            continue;
        }
        float acc[kUnroll][8];
#pragma unroll
        for (int j = 0; j < kUnroll; ++j)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[j][i] = 0.0f;
        bool in_row[kUnroll];
#pragma unroll
        for (int j = 0; j < kUnroll; ++j) in_row[j] = col0 + j * kColBytes < a.row_bytes;
        if (KT > 0) {
            uint4 v[kUnroll][KR];
#pragma unroll
            for (int j = 0; j < kUnroll; ++j)
#pragma unroll
                for (int k = 0; k < KR; ++k) v[j][k] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int k = 0; k < KR; ++k)
#pragma unroll
                for (int j = 0; j < kUnroll; ++j)
                    if (on[k] && in_row[j]) v[j][k] = ld_nc_v4_dep(row(k) + col0 + j * kColBytes);
#pragma unroll
            for (int j = 0; j < kUnroll; ++j)
#pragma unroll
                for (int k = 0; k < KR; ++k)
                    if (on[k] && in_row[j]) fma8(acc[j], wk[k], v[j][k]);
        } else {
            // Any K <= 32, kGenericBatch entries of k at a time: all their
            // loads are issued before their fmas, which still run in k order.
            for (int k0 = 0; k0 < K; k0 += kGenericBatch) {
                uint4 v[kUnroll][kGenericBatch];
                float wq[kGenericBatch];
                bool onq[kGenericBatch];
#pragma unroll
                for (int q = 0; q < kGenericBatch; ++q) {
                    const int k = k0 + q;  // < 32 + kGenericBatch; lanes read mod 32
                    const int32_t sk = __shfl_sync(kFullMask, s_lane, k & 31);
                    wq[q] = __shfl_sync(kFullMask, w_lane, k & 31);
                    onq[q] = k < K && sk >= 0;
                    const uint8_t* row =
                        a.expert_out + static_cast<int64_t>(onq[q] ? sk : 0) * a.row_bytes;
#pragma unroll
                    for (int j = 0; j < kUnroll; ++j)
                        v[j][q] = (onq[q] && in_row[j]) ? ld_nc_v4_dep(row + col0 + j * kColBytes)
                                                        : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int q = 0; q < kGenericBatch; ++q)
#pragma unroll
                    for (int j = 0; j < kUnroll; ++j)
                        if (onq[q] && in_row[j]) fma8(acc[j], wq[q], v[j][q]);
            }
        }
        uint8_t* yrow = a.y + t * static_cast<int64_t>(a.row_bytes);
#pragma unroll
        for (int j = 0; j < kUnroll; ++j)
            if (in_row[j]) st_v4(yrow + col0 + j * kColBytes, round8(acc[j]));
        if (++cb == n_cb) {
            cb = 0;
            ++t;
        }
    }
}

template <int KT, int kThreads, int kUnroll, bool kFast, bool kSlotRows>
cudaError_t launch_shape(const CombineArgs& a, int num_sms, cudaStream_t stream) {
    constexpr uint32_t kUnitBytes = kColBytes * kUnroll;
    const int64_t units = a.T * ((a.row_bytes + kUnitBytes - 1) / kUnitBytes);
    const int64_t warps_per_cta = kThreads / 32;
    // a.tail_percent of the units to a tail launch (as dispatch's: small
    // CTAs that start on SMs as the persistent CTAs leave them; a combine
    // CTA holds the whole register file, so nothing shares its SM)
    const int64_t tail = units * a.tail_percent / 100;
    CombineArgs main = a;
    main.unit_base = 0;
    main.unit_count = units - tail;
    const int64_t ctas_needed = (main.unit_count + warps_per_cta - 1) / warps_per_cta;
    const int grid = static_cast<int>(ctas_needed < num_sms ? ctas_needed : num_sms);
    if (grid <= 0) return cudaSuccess;
    auto kern = combine_kernel<KT, kThreads, kUnroll, kFast, kSlotRows>;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(kExclusiveSmem));
    if (err != cudaSuccess) return err;
    err = launch_dependent(kern, grid, kThreads, kExclusiveSmem, stream, main);
    if (err != cudaSuccess || tail <= 0) return err;
    CombineArgs t = a;
    t.unit_base = main.unit_count;
    t.unit_count = tail;
    t.tail = 1;
    constexpr int kTailThreads = EP_COMBINE_TAIL_WARPS * 32;
    const int64_t per_cta = static_cast<int64_t>(EP_COMBINE_TAIL_WARPS) * EP_COMBINE_TAIL_UNITS;
    const int tail_grid = static_cast<int>((tail + per_cta - 1) / per_cta);
    return launch_dependent(kern, tail_grid, kTailThreads, 0, stream, t);
}

// CTAs a shape needs for one unit per warp.
int64_t ctas_for_shape(const CombineArgs& a, int threads, int unroll) {
    const int64_t unit_bytes = static_cast<int64_t>(kColBytes) * unroll;
    const int64_t units = a.T * ((a.row_bytes + unit_bytes - 1) / unit_bytes);
    const int64_t warps = threads / 32;
    return (units + warps - 1) / warps;
}

template <int KT>
cudaError_t launch_k(const CombineArgs& a, int num_sms, cudaStream_t stream) {
    constexpr CombineShape c = combine_shape(KT);
    const bool small = KT == 0 ? num_sms >= kGenericWideSms
                               : ctas_for_shape(a, c.threads, c.unroll) < num_sms;
    if (small)
        return launch_shape<KT, kSmallThreads, kSmallUnroll, (KT > 0), false>(a, num_sms, stream);
    return launch_shape<KT, c.threads, c.unroll, (KT > 0), c.slot_rows>(a, num_sms, stream);
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, int num_sms, cudaStream_t stream) {
    switch (a.K) {
        case 1: return launch_k<1>(a, num_sms, stream);
        case 2: return launch_k<2>(a, num_sms, stream);
        case 3: return launch_k<3>(a, num_sms, stream);
        case 4: return launch_k<4>(a, num_sms, stream);
        case 5: return launch_k<5>(a, num_sms, stream);
        case 6: return launch_k<6>(a, num_sms, stream);
        case 7: return launch_k<7>(a, num_sms, stream);
        case 8: return launch_k<8>(a, num_sms, stream);
        default: return launch_k<0>(a, num_sms, stream);
    }
}

}  // namespace ep
