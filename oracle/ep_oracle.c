/*
 * ep_oracle.c -- CPU oracle for MoE dispatch / combine data movement.
 *
 * TEST INFRASTRUCTURE ONLY (see ep_oracle.h). Single thread, no SIMD, no
 * blocking or reordering: each function is the plain definition written out.
 * Build: cc -O2 -ffp-contract=off -fPIC -shared (contraction off, so every
 * multiply-add in combine is the explicit fmaf call and nothing else).
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one known mistake. It exists
 * only so the test suite can show that its pins catch plausible errors; the
 * library the tests and benchmark load is always built with ORACLE_MUTANT=0.
 */
#include "ep_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---- bf16 <-> fp32 ------------------------------------------------------
 * bf16 keeps the sign, the 8 exponent bits and the top 7 fraction bits of an
 * IEEE-754 binary32. Widening is exact: append 16 zero bits. Narrowing rounds
 * to nearest, ties to even: add 0x7FFF plus the lowest kept bit, then drop
 * the low 16 bits (a carry into the exponent is the correct round-up, up to
 * and including overflow to infinity). NaN stays NaN (quiet bit forced). */
float oracle_bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t oracle_f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);           /* NaN -> quiet NaN */
#if ORACLE_MUTANT == 6
    return (uint16_t)(u >> 16);                           /* planted: truncation */
#else
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
#endif
}

/* ---- layout ----------------------------------------------------------------
 * Entry (t,k) goes to expert e = idx[t,k]. counts is the histogram over the
 * valid entries, offsets its exclusive prefix (offsets[E] = total), and the
 * entries of expert e occupy rows offsets[e] .. offsets[e+1]-1 of the receive
 * buffer in ascending (t, k) order. */
int oracle_layout(const int64_t* topk_idx, int64_t T, int K, int E,
                  int32_t* counts, int32_t* offsets, int32_t* slot) {
    int status = ORACLE_OK;
    int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)(E > 0 ? E : 1));
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (int64_t t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[t * K + k];
            if (e >= 0 && e < E) {
                counts[e] += 1;
            } else if (e != -1) {
                status = ORACLE_BAD_EXPERT;
            }
        }
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
#if ORACLE_MUTANT == 4
        offsets[e + 1] = offsets[e] + counts[e] + (e == 0);  /* planted: off by one */
#else
        offsets[e + 1] = offsets[e] + counts[e];
#endif
    }
    for (int e = 0; e < E; ++e) fill[e] = offsets[e];
#if ORACLE_MUTANT == 3
    for (int64_t t = T - 1; t >= 0; --t) {                 /* planted: unstable order */
#else
    for (int64_t t = 0; t < T; ++t) {
#endif
        for (int k = 0; k < K; ++k) {
            int64_t e = topk_idx[t * K + k];
            if (e >= 0 && e < E) {
                slot[t * K + k] = fill[e];
                fill[e] += 1;
            } else {
                slot[t * K + k] = -1;
            }
        }
    }
    free(fill);
    return status;
}

/* ---- dispatch -------------------------------------------------------------
 * The receive loop of [DeepEP-TMA] "Asynchronous Copy Primitives" copies each
 * received token row into its slot of the receive buffer; on one GPU that is
 * a plain row copy per valid (t,k). */
void oracle_dispatch(const uint16_t* x, int64_t T, int64_t H, int K,
                     const int32_t* slot, const float* topk_w,
                     uint16_t* recv_x, float* recv_w, int32_t* recv_src) {
    for (int64_t t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k) {
            int32_t s = slot[t * K + k];
            if (s < 0) continue;
#if ORACLE_MUTANT == 5
            int64_t src = (t + 1) % T;                     /* planted: wrong row */
#else
            int64_t src = t;
#endif
            memcpy(recv_x + (int64_t)s * H, x + src * H, sizeof(uint16_t) * (size_t)H);
            if (recv_w) recv_w[s] = topk_w[t * K + k];
            if (recv_src) recv_src[s] = (int32_t)(t * K + k);
        }
    }
}

/* ---- combine --------------------------------------------------------------
 * Gather each token's K expert rows back and reduce them with the routing
 * weights: fp32 accumulator from +0.0f, one fused multiply-add per k in
 * ascending k, a single bf16 rounding at the end. */
void oracle_combine(const uint16_t* expert_out, const int32_t* slot,
                    const float* topk_w, int64_t T, int64_t H, int K,
                    uint16_t* y) {
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
#if ORACLE_MUTANT == 1
            for (int k = 0; k < K - 1; ++k) {              /* planted: last term dropped */
#elif ORACLE_MUTANT == 10
            for (int k = K - 1; k >= 0; --k) {             /* planted: descending k */
#else
            for (int k = 0; k < K; ++k) {
#endif
                int32_t s = slot[t * K + k];
                if (s < 0) continue;
#if ORACLE_MUTANT == 2
                float w = topk_w[t * K + (K - 1 - k)];     /* planted: weight index reversed */
#else
                float w = topk_w[t * K + k];
#endif
                float v = oracle_bf16_to_f32(expert_out[(int64_t)s * H + h]);
#if ORACLE_MUTANT == 7
                acc = fmaf(w, v, -acc);                    /* planted: sign error */
#elif ORACLE_MUTANT == 9
                acc = acc + w * v;                         /* planted: two roundings */
#else
                acc = fmaf(w, v, acc);
#endif
            }
            y[t * H + h] = oracle_f32_to_bf16_rne(acc);
        }
    }
}

/* ---- two-stage pipeline model ------------------------------------------
 * [TMA-atlas] "Science and assumptions": after the first tile has been both
 * loaded and computed, each of the remaining N-1 tiles costs one interval of
 * the slower stage. Without overlap the N tiles cost N * (t_load + t_compute). */
double oracle_pipeline_time(int64_t N, double t_load, double t_compute) {
    if (N <= 0) return 0.0;
#if ORACLE_MUTANT == 8
    double slower = t_load < t_compute ? t_load : t_compute;  /* planted: min */
#else
    double slower = t_load > t_compute ? t_load : t_compute;
#endif
    return t_load + t_compute + (double)(N - 1) * slower;
}

double oracle_serial_time(int64_t N, double t_load, double t_compute) {
    if (N <= 0) return 0.0;
    return (double)N * (t_load + t_compute);
}
