// MX (OCP microscaling) quantiser used on the device: the activation
// quantiser before stage 1 and the requantiser in the stage-1 epilogue.
#pragma once

#include <stdint.h>

namespace moe {

// ============================================================== MX quantiser
//
// OCP MX rule with 32-element blocks (the activation quantiser the pages call
// in kernelbot-amd-moe-mxfp4-754773, flower_moe.py, custom_kernel):
//   s = e8m0 byte of 2^X, X = floor(log2 amax) - 2 clamped to [-127, 127];
//   element = sign | nearest e2m1 magnitude of |v| * 2^-X, ties to the even
//   mantissa bit, saturating at 6.  A NaN/Inf in the block gives s = 255 and
//   signed zeros.  Shared by the quant kernel and the stage-1 epilogue.

// Scale byte of a block from the bit pattern of its amax (sign bit clear).
__device__ __forceinline__ uint32_t mx_scale_byte(uint32_t amax_bits) {
    if (amax_bits >= 0x7f800000u) return 255u;
    const int e = (int)(amax_bits >> 23);  // biased exponent; 0 for zero/subnormal
    const int s = e - 2;                   // X + 127 with X = (e - 127) - 2
    return (uint32_t)(s < 0 ? 0 : s);
}

// 2^-X for a finite scale byte s (X = s - 127): exponent field 254 - s.
__device__ __forceinline__ float mx_inv_scale(uint32_t s) {
    return __uint_as_float((254u - s) << 23);
}

// e2m1 magnitude code of q >= 0 (round to nearest, ties to even, saturate).
__device__ __forceinline__ uint32_t e2m1_mag(float q) {
    return (uint32_t)(q > 0.25f) + (uint32_t)(q >= 0.75f) + (uint32_t)(q > 1.25f) +
           (uint32_t)(q >= 1.75f) + (uint32_t)(q > 2.5f) + (uint32_t)(q >= 3.5f) +
           (uint32_t)(q > 5.0f);
}

__device__ __forceinline__ uint32_t e2m1_code(float v, uint32_t s, float inv) {
    const uint32_t sign = (__float_as_uint(v) >> 31) << 3;
    if (s == 255u) return sign;
    return sign | e2m1_mag(fabsf(v) * inv);
}

}  // namespace moe
