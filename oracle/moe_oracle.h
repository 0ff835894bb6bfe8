/*
 * CPU oracle for the fused MXFP4 Mixture-of-Experts forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code: it exists so that tests/, the smoke check and the CPU
 * baseline of the benchmark can compare the CUDA library against a plain,
 * slow, obviously correct restatement of the method.  It shares no code,
 * header, table or constant with the CUDA sources.
 *
 * Sources (web pages; "solution.py" and "flower_moe.py" are the code listings
 * printed on the pages):
 *   [P1] kernelbot-amd-moe-mxfp4-754773, flower_moe.py
 *        - _flower_get_sort_buffers (sorted-buffer capacity),
 *        - custom_kernel (sort -> quant(hidden) -> stage1 -> quant(a2) -> stage2).
 *   [P2] kernelbot-amd-moe-mxfp4-723815, solution.py
 *        - fp4_to_f32 / e8m0_to_f32 / _dequant (element and scale decoding, nibble order),
 *        - kernel_stage1 / kernel_stage2 / _reference_forward (gate/up layout, SwiGLU,
 *          down projection, top-k weight after the down GEMM),
 *        - _make (tensor shapes).
 *   [P3] b12x moe/fused/w4a16/kernel.py
 *        - route index t*topk+k, sentinel = T*topk for padding (_read_moe_block_data).
 *   The activation quantiser follows the OCP MX rule (shared exponent
 *   floor(log2(amax)) - 2, round to nearest even on the e2m1 grid, clamp +-6);
 *   the pages only call that kernel, they do not print it.
 *
 * Precision: fp32 everywhere on the method's path, as the pages fix it (fp32
 * accumulators in kernel_stage1/kernel_stage2, bf16 intermediate a2 in
 * flower_moe.py, bf16 output).  Build with -ffp-contract=off so that no
 * multiply-add is fused.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Value of a 4-bit e2m1 code (bit 3 sign, bits 2..1 exponent, bit 0 mantissa). */
float moe_oracle_e2m1(int code);

/* Value of an e8m0 scale byte: 2^(s-127); s = 255 (NaN in OCP MX) returns NaN. */
float moe_oracle_e8m0(int s);

/* Round an fp32 value to the nearest bf16 (ties to even), returned as bits. */
uint16_t moe_oracle_bf16_bits(float x);

/* fp32 value of a bf16 bit pattern. */
float moe_oracle_bf16_value(uint16_t bits);

/*
 * MX quantiser for one block of 32 values.
 *   codes: 16 bytes, element 2i in the low nibble of byte i, 2i+1 in the high nibble.
 *   scale: one e8m0 byte.
 */
void moe_oracle_quant_block(const float* v, uint8_t* codes, uint8_t* scale);

/* Quantise a row of n values (n % 32 == 0): n/2 code bytes and n/32 scale bytes. */
void moe_oracle_quant_row(const float* v, int n, uint8_t* codes, uint8_t* scales);

/* Capacity of the padded sorted arrays for R = T*topk routes, E experts, block bm. */
int moe_oracle_route_capacity(int T, int topk, int E, int bm);

/*
 * Routing: group routes r = t*topk + k by expert, ascending r within an expert,
 * each expert's segment padded with the sentinel R to a multiple of bm.
 *   sorted_ids   [cap]          route id or R (padding / unused tail)
 *   sorted_w     [cap]          topk_weights[route] or 0
 *   block_expert [cap/bm]       expert of each bm-block, -1 past the used blocks
 *   seg_start    [E+1]          start of each expert's segment; seg_start[E] = padded length
 *   route_pos    [R]            position of route r in sorted_ids, -1 for ids outside [0,E)
 *   num_valid    [2]            { padded length, number of valid routes }
 * Returns 0, or -1 when cap is too small.
 */
int moe_oracle_route(const int32_t* topk_ids, const float* topk_w, int T, int topk, int E,
                     int bm, int cap, int32_t* sorted_ids, float* sorted_w,
                     int32_t* block_expert, int32_t* seg_start, int32_t* route_pos,
                     int32_t* num_valid);

/*
 * Forward pass for the tokens listed in `tokens` (all T tokens when tokens == NULL).
 *   hidden    bf16 bits [T, D]
 *   w13       [E, 2I, D/2] packed e2m1 (rows 0..I-1 gate, I..2I-1 up), w13s [E, 2I, D/32]
 *   w2        [E, D, I/2] packed e2m1, w2s [E, D, I/32]
 *   topk_ids  [T, K], topk_w [T, K]
 * Outputs (rows of tokens not in the subset are left untouched; any may be NULL):
 *   a1q [T, D/2], a1s [T, D/32]      quantised hidden rows
 *   h   [T*K, I]                      bf16-rounded SwiGLU output per route (as fp32)
 *   a2q [T*K, I/2], a2s [T*K, I/32]  quantised h per route
 *   out_f32 [T, D]                    top-k weighted sum before the final rounding
 *   out_bf16 [T, D]                   bf16 bits of out_f32
 * quant_act = 1 runs the method (MXFP4 activations); 0 keeps hidden and h in
 * fp32/bf16 without the two activation quantisations (the W4A16 reading used
 * by the page's pure-PyTorch reference).
 * n_threads <= 1 runs single-threaded; results do not depend on n_threads.
 * Returns 0, or -1 on a bad argument.
 */
int moe_oracle_forward(const uint16_t* hidden, const uint8_t* w13, const uint8_t* w13s,
                       const uint8_t* w2, const uint8_t* w2s, const int32_t* topk_ids,
                       const float* topk_w, int T, int D, int I, int E, int K,
                       const int32_t* tokens, int n_tokens, int quant_act,
                       uint8_t* a1q, uint8_t* a1s, float* h, uint8_t* a2q, uint8_t* a2s,
                       float* out_f32, uint16_t* out_bf16, int n_threads);

/* Number of OpenMP threads available (1 when built without OpenMP). */
int moe_oracle_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
