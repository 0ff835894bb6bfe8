/*
 * CPU oracle for the fused MXFP4 Mixture-of-Experts forward.
 *
 * TEST INFRASTRUCTURE ONLY (see moe_oracle.h): called by tests/, the smoke
 * check and the CPU-baseline leg of bench.py, never by the product path.
 *
 * Every function restates one step of the method in the plainest form, in the
 * order the pages give it, in fp32.  No blocking, fusion or reordering: each
 * output element is a single ascending loop, so the result does not depend on
 * the number of threads.  Compile with -ffp-contract=off.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------- decoding */

/*
 * e2m1 element: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
 * Exponent field 0 is subnormal: value = mantissa * 0.5.  Otherwise
 * value = (1 + mantissa/2) * 2^(exponent - 1).
 * [P2] kernelbot-amd-moe-mxfp4-723815, solution.py: fp4_to_f32 and _dequant.
 */
float moe_oracle_e2m1(int code) {
    int sign = (code >> 3) & 1;
    int expo = (code >> 1) & 3;
    int mant = code & 1;
    float mag;
    if (expo == 0)
        mag = 0.5f * (float)mant;
    else
        mag = ldexpf(1.0f + 0.5f * (float)mant, expo - 1);
    return sign ? -mag : mag;
}

/*
 * e8m0 scale: an unbiased power of two, 2^(s - 127).
 * [P2] solution.py: e8m0_to_f32 and the `2.0 ** (scale - 127)` step of _dequant.
 * OCP MX reserves s = 255 for NaN.
 */
float moe_oracle_e8m0(int s) {
    if (s == 255) return NAN;
    return ldexpf(1.0f, s - 127);
}

/* Round-to-nearest-even fp32 -> bf16 (the bf16 a2 buffer of [P1] custom_kernel
 * and the bf16 output). NaN stays NaN. */
uint16_t moe_oracle_bf16_bits(float x) {
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

float moe_oracle_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ---------------------------------------------------------------- quantiser */

/*
 * Round a magnitude m (finite, >= 0) to the e2m1 grid {0, .5, 1, 1.5, 2, 3, 4, 6}:
 * nearest grid value, ties to the value whose mantissa bit is 0 (even code),
 * values above 6 saturate to 6.  Returns the 3-bit magnitude code.
 */
static int e2m1_round_magnitude(float m) {
    if (m >= 6.0f) return 7;
    int best = 0;
    double dbest = fabs((double)m - (double)moe_oracle_e2m1(0));
    for (int i = 1; i < 8; ++i) {
        double d = fabs((double)m - (double)moe_oracle_e2m1(i));
        if (d < dbest || (d == dbest && (i & 1) == 0)) {
            best = i;
            dbest = d;
        }
    }
    return best;
}

/*
 * OCP MX quantisation of one block of 32 fp32 values:
 *   amax = max |v_i|;  X = floor(log2(amax)) - 2 (2 = largest e2m1 exponent),
 *   clamped to the e8m0 range [-127, 127];  scale byte s = X + 127;
 *   element code = sign(v_i) | round_even(|v_i| / 2^X), saturating at 6.
 * Readings (the pages call this kernel without printing it):
 *   - amax == 0: X clamps to -127 (s = 0) and every element is a signed zero;
 *   - a NaN/Inf in the block: s = 255 (e8m0 NaN) and every element a signed zero;
 *   - the sign bit is kept for elements that round to zero (-0 -> code 8).
 * floor(log2(amax)) is read from the fp32 exponent (frexpf), with no log2f.
 */
void moe_oracle_quant_block(const float* v, uint8_t* codes, uint8_t* scale) {
    float amax = 0.0f;
    int finite = 1;
    for (int i = 0; i < 32; ++i) {
        if (!isfinite(v[i])) finite = 0;
        float a = fabsf(v[i]);
        if (a > amax) amax = a;
    }
    memset(codes, 0, 16);
    if (!finite) {
        *scale = 255;
        for (int i = 0; i < 32; ++i) {
            int c = signbit(v[i]) ? 8 : 0;
            codes[i / 2] |= (uint8_t)(c << (4 * (i & 1)));
        }
        return;
    }
    int X;
    if (amax == 0.0f) {
        X = -127;
    } else {
        int e;
        frexpf(amax, &e); /* amax = f * 2^e, f in [0.5, 1) => floor(log2 amax) = e - 1 */
        X = (e - 1) - 2;
        if (X < -127) X = -127;
        if (X > 127) X = 127;
    }
    *scale = (uint8_t)(X + 127);
    for (int i = 0; i < 32; ++i) {
        float q = ldexpf(v[i], -X); /* exact: division by a power of two */
        int c = e2m1_round_magnitude(fabsf(q));
        if (signbit(v[i])) c |= 8;
        codes[i / 2] |= (uint8_t)(c << (4 * (i & 1)));
    }
}

void moe_oracle_quant_row(const float* v, int n, uint8_t* codes, uint8_t* scales) {
    for (int b = 0; b < n / 32; ++b) moe_oracle_quant_block(v + 32 * b, codes + 16 * b, scales + b);
}

/* ---------------------------------------------------------------- routing */

/*
 * Capacity of the padded sorted arrays: every expert that has at least one
 * route adds fewer than bm padding slots, and at most min(E, R) experts have
 * a route; rounded up to a whole block.  (Same role as max_padded in
 * [P1] _flower_get_sort_buffers.)
 */
int moe_oracle_route_capacity(int T, int topk, int E, int bm) {
    long R = (long)T * topk;
    long used = R < E ? R : E;
    long cap = R + used * (bm - 1);
    cap = (cap + bm - 1) / bm * bm;
    return (int)cap;
}

/*
 * Counting sort of routes by expert.  [P2] kernel_count_tokens /
 * kernel_prefix_sum / kernel_scatter_tokens give the count -> prefix -> scatter
 * structure; [P1] custom_kernel gives the block_m padding and per-block expert
 * ids; [P3] _read_moe_block_data gives the route index t*topk+k and the
 * sentinel T*topk.  Reading: routes appear in ascending route id within an
 * expert (the pages' atomic cursor leaves that order unspecified); ids
 * outside [0, E) are skipped, as kernel_count_tokens does.
 */
int moe_oracle_route(const int32_t* topk_ids, const float* topk_w, int T, int topk, int E,
                     int bm, int cap, int32_t* sorted_ids, float* sorted_w,
                     int32_t* block_expert, int32_t* seg_start, int32_t* route_pos,
                     int32_t* num_valid) {
    int R = T * topk;
    if (bm <= 0 || E <= 0 || cap % bm != 0) return -1;
    int32_t* cnt = (int32_t*)calloc((size_t)E, sizeof(int32_t));
    if (!cnt) return -1;
    int valid = 0;
    for (int r = 0; r < R; ++r) {
        int e = topk_ids[r];
        if (e >= 0 && e < E) {
            cnt[e] += 1;
            valid += 1;
        }
    }
    seg_start[0] = 0;
    for (int e = 0; e < E; ++e) seg_start[e + 1] = seg_start[e] + (cnt[e] + bm - 1) / bm * bm;
    free(cnt);
    if (seg_start[E] > cap) return -1;

    for (int p = 0; p < cap; ++p) {
        sorted_ids[p] = R;
        sorted_w[p] = 0.0f;
    }
    for (int b = 0; b < cap / bm; ++b) block_expert[b] = -1;
    for (int r = 0; r < R; ++r) route_pos[r] = -1;

    for (int e = 0; e < E; ++e) {
        int p = seg_start[e];
        for (int r = 0; r < R; ++r) {
            if (topk_ids[r] == e) {
                sorted_ids[p] = r;
                sorted_w[p] = topk_w[r];
                route_pos[r] = p;
                ++p;
            }
        }
        for (int b = seg_start[e] / bm; b < seg_start[e + 1] / bm; ++b) block_expert[b] = e;
    }
    num_valid[0] = seg_start[E];
    num_valid[1] = valid;
    return 0;
}

/* ---------------------------------------------------------------- forward */

/* Value tables filled from moe_oracle_e2m1 / moe_oracle_e8m0 (a cache of the
 * two definitions above, so the inner loops do not call ldexpf). */
static float g_e2m1[16];
static float g_e8m0[256];

static void fill_tables(void) {
    for (int c = 0; c < 16; ++c) g_e2m1[c] = moe_oracle_e2m1(c);
    for (int s = 0; s < 256; ++s) g_e8m0[s] = moe_oracle_e8m0(s);
}

/* Decode one packed row of n e2m1 elements with n/32 e8m0 scales into fp32.
 * Byte j holds element 2j in its low nibble and 2j+1 in its high nibble
 * ([P2] _dequant: stack(lo, hi)). Each value code * 2^(s-127) is exact. */
static void dequant_row(const uint8_t* codes, const uint8_t* scales, int n, float* outv) {
    for (int j = 0; j < n; ++j) {
        int byte = codes[j / 2];
        int nib = (j & 1) ? (byte >> 4) & 15 : byte & 15;
        outv[j] = g_e2m1[nib] * g_e8m0[scales[j / 32]];
    }
}

/* fp32 dot product accumulated in ascending index order. */
static float dot_f32(const float* a, const float* b, int n) {
    float acc = 0.0f;
    for (int j = 0; j < n; ++j) acc = acc + a[j] * b[j];
    return acc;
}

int moe_oracle_forward(const uint16_t* hidden, const uint8_t* w13, const uint8_t* w13s,
                       const uint8_t* w2, const uint8_t* w2s, const int32_t* topk_ids,
                       const float* topk_w, int T, int D, int I, int E, int K,
                       const int32_t* tokens, int n_tokens, int quant_act,
                       uint8_t* a1q, uint8_t* a1s, float* h, uint8_t* a2q, uint8_t* a2s,
                       float* out_f32, uint16_t* out_bf16, int n_threads) {
    if (T < 0 || D <= 0 || I <= 0 || E <= 0 || K <= 0 || D % 32 || I % 32) return -1;
    if (tokens == NULL) n_tokens = T;
    for (int i = 0; i < n_tokens; ++i) {
        int t = tokens ? tokens[i] : i;
        if (t < 0 || t >= T) return -1;
    }
    if (n_threads < 1) n_threads = 1;
    int bad = 0;
    fill_tables();

#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(n_threads)
#endif
    for (int i = 0; i < n_tokens; ++i) {
        int t = tokens ? tokens[i] : i;
        float* x = (float*)malloc(sizeof(float) * (size_t)D);
        float* wrow = (float*)malloc(sizeof(float) * (size_t)(D > I ? D : I));
        float* wrow2 = (float*)malloc(sizeof(float) * (size_t)D);
        float* hv = (float*)malloc(sizeof(float) * (size_t)I);
        float* av = (float*)malloc(sizeof(float) * (size_t)I);
        float* acc = (float*)malloc(sizeof(float) * (size_t)D);
        uint8_t* qc = (uint8_t*)malloc((size_t)(D > I ? D : I) / 2);
        uint8_t* qs = (uint8_t*)malloc((size_t)(D > I ? D : I) / 32);
        if (!x || !wrow || !wrow2 || !hv || !av || !acc || !qc || !qs) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            bad = 1;
            free(x); free(wrow); free(wrow2); free(hv); free(av); free(acc); free(qc); free(qs);
            continue;
        }

        /* Activation of token t: bf16 hidden row, quantised per token once
         * ([P1] custom_kernel quantises hidden_states with topk=1). */
        for (int j = 0; j < D; ++j) x[j] = moe_oracle_bf16_value(hidden[(size_t)t * D + j]);
        if (quant_act) {
            moe_oracle_quant_row(x, D, qc, qs);
            if (a1q) memcpy(a1q + (size_t)t * (D / 2), qc, (size_t)D / 2);
            if (a1s) memcpy(a1s + (size_t)t * (D / 32), qs, (size_t)D / 32);
            dequant_row(qc, qs, D, x);
        }

        for (int n = 0; n < D; ++n) acc[n] = 0.0f;

        for (int k = 0; k < K; ++k) {
            size_t r = (size_t)t * K + k;
            int e = topk_ids[r];
            if (e < 0 || e >= E) continue; /* contributes nothing */

            /* Stage 1: gate rows [0, I), up rows [I, 2I) of w13[e]
             * ([P2] kernel_stage1, _reference_forward: W_gate / W_up). */
            const uint8_t* w13e = w13 + (size_t)e * 2 * I * (D / 2);
            const uint8_t* w13se = w13s + (size_t)e * 2 * I * (D / 32);
            for (int n = 0; n < I; ++n) {
                dequant_row(w13e + (size_t)n * (D / 2), w13se + (size_t)n * (D / 32), D, wrow);
                float g = dot_f32(x, wrow, D);
                dequant_row(w13e + (size_t)(I + n) * (D / 2), w13se + (size_t)(I + n) * (D / 32), D,
                            wrow2);
                float u = dot_f32(x, wrow2, D);
                /* SwiGLU: silu(g) * u with silu(g) = g / (1 + e^-g) ([P2] silu). */
                float s = g / (1.0f + expf(-g));
                float v = s * u;
                hv[n] = moe_oracle_bf16_value(moe_oracle_bf16_bits(v)); /* bf16 a2 buffer */
            }
            if (h) memcpy(h + r * I, hv, sizeof(float) * (size_t)I);

            /* Requantise the intermediate per route ([P1] custom_kernel, second quant). */
            if (quant_act) {
                moe_oracle_quant_row(hv, I, qc, qs);
                if (a2q) memcpy(a2q + r * (I / 2), qc, (size_t)I / 2);
                if (a2s) memcpy(a2s + r * (I / 32), qs, (size_t)I / 32);
                dequant_row(qc, qs, I, av);
            } else {
                memcpy(av, hv, sizeof(float) * (size_t)I);
            }

            /* Stage 2: y = W2[e] . a, then the top-k weight, summed over k in
             * ascending order ([P2] kernel_stage2: the weight multiplies the
             * down-projection output; [P1] stage2 takes sorted_weights). */
            const uint8_t* w2e = w2 + (size_t)e * D * (I / 2);
            const uint8_t* w2se = w2s + (size_t)e * D * (I / 32);
            float wk = topk_w[r];
            for (int n = 0; n < D; ++n) {
                dequant_row(w2e + (size_t)n * (I / 2), w2se + (size_t)n * (I / 32), I, wrow);
                float y = dot_f32(av, wrow, I);
                float p = wk * y;
                acc[n] = acc[n] + p;
            }
        }

        for (int n = 0; n < D; ++n) {
            if (out_f32) out_f32[(size_t)t * D + n] = acc[n];
            if (out_bf16) out_bf16[(size_t)t * D + n] = moe_oracle_bf16_bits(acc[n]);
        }
        free(x); free(wrow); free(wrow2); free(hv); free(av); free(acc); free(qc); free(qs);
    }
    return bad ? -1 : 0;
}

int moe_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
