/*
 * ep_oracle.h -- CPU oracle for MoE dispatch / combine data movement.
 *
 * TEST INFRASTRUCTURE ONLY. This is a plain, slow, single-threaded C
 * restatement of what the GPU path computes. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it. It shares no code,
 * header, table or helper with the CUDA library.
 *
 * Sources (web pages studied):
 *  [DeepEP-TMA]  "How DeepEP Utilizes TMA Instructions for Minimal SM Usage on
 *                Hopper GPUs" (instagit.com deep-dive).
 *  [TMA-atlas]   "tensor-memory-accelerator" (semiaifoundry.com atlas).
 *
 * The pages show only DeepEP's dispatch call and its receive loop; they do
 * not describe the layout step or combine. Those follow the plainest reading
 * of the problem (each token's row goes to each of its top-k experts'
 * contiguous receive segments; combine is the weighted inverse gather), as
 * listed in the readings of the design notes:
 *   - rows inside an expert segment are in ascending (t, k) order (stable);
 *   - topk_idx == -1 masks an entry (slot -1, skipped everywhere);
 *   - any other id outside [0, E) is skipped and reported as ORACLE_BAD_EXPERT;
 *   - combine: acc = +0.0f, then acc = fmaf(w[t,k], float(e[slot,h]), acc)
 *     for k = 0..K-1 ascending, skipping slot < 0, then one bf16
 *     round-to-nearest-even.
 *
 * Parity pins: every function here is pinned by the not-gpu tests (library
 * routines, closed forms, brute force, the pages' worked example).
 */
#ifndef EP_ORACLE_H
#define EP_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_EXPERT 5

/* bf16 <-> fp32 by bit manipulation (bf16 = upper 16 bits of an IEEE fp32). */
float    oracle_bf16_to_f32(uint16_t b);
uint16_t oracle_f32_to_bf16_rne(float f);

/* Layout: counts[e] = #{(t,k) : idx[t,k] == e}; offsets = exclusive prefix
 * of counts with offsets[E] = number of valid entries; slot[t,k] = position
 * of (t,k) in the expert-major, (t,k)-stable receive order, -1 if masked or
 * invalid. Returns ORACLE_OK or ORACLE_BAD_EXPERT. */
int oracle_layout(const int64_t* topk_idx, int64_t T, int K, int E,
                  int32_t* counts, int32_t* offsets, int32_t* slot);

/* Dispatch: recv_x[slot[t,k]] = x[t] (H bf16 values) for every valid (t,k);
 * recv_w[slot] = topk_w[t,k] and recv_src[slot] = t*K+k when those outputs
 * are non-NULL. */
void oracle_dispatch(const uint16_t* x, int64_t T, int64_t H, int K,
                     const int32_t* slot, const float* topk_w,
                     uint16_t* recv_x, float* recv_w, int32_t* recv_src);

/* Combine: y[t,h] = bf16_rne( fma chain over k ascending of
 * topk_w[t,k] * float(expert_out[slot[t,k], h]) ), chain starting at +0.0f,
 * entries with slot < 0 skipped. */
void oracle_combine(const uint16_t* expert_out, const int32_t* slot,
                    const float* topk_w, int64_t T, int64_t H, int K,
                    uint16_t* y);

/* Two-stage pipeline closed form of [TMA-atlas] "Science and assumptions":
 * first load + first compute, then N-1 intervals set by the slower stage. */
double oracle_pipeline_time(int64_t N, double t_load, double t_compute);
/* The same N tiles without overlap: N * (t_load + t_compute). */
double oracle_serial_time(int64_t N, double t_load, double t_compute);

#ifdef __cplusplus
}
#endif
#endif
