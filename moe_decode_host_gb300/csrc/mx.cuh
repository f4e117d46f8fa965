// MXFP4 conversion of activations (the OCP Microscaling rule for E2M1 elements),
// shared by the stand-alone quantiser and the block-scaled prefill kernels: each
// 32-element block gets the exponent floor(log2(max |v|)) - 2 (2 = the exponent of
// E2M1's largest value, 6 = 1.5 * 2^2), clamped to the E8M0 range [-127, 127] (an
// all-zero block takes -127); each element gets |v| / 2^exp rounded to the nearest
// E2M1 magnitude {0, 0.5, 1, 1.5, 2, 3, 4, 6}, ties to the even code, above 6
// saturating to 6, with v's sign bit.
#pragma once

#include <stdint.h>

namespace moe {

// floor(log2(a)) of a positive finite float given by its bits.
__device__ __forceinline__ int floor_log2_bits(uint32_t b) {
    const int ef = (int)((b >> 23) & 0xffu);
    if (ef != 0) return ef - 127;
    const uint32_t m = b & 0x7fffffu;  // subnormal: m * 2^-149, m != 0
    return (31 - __clz((int)m)) - 149;
}

// Shared block exponent from the largest magnitude's bits (0 for an all-zero block).
__device__ __forceinline__ int mx_block_exp(uint32_t amax_bits) {
    return amax_bits == 0u ? -127 : max(-127, min(127, floor_log2_bits(amax_bits) - 2));
}

// |v| / 2^e for the bits of |v| and a block exponent e of its block: exact (a
// power-of-two scaling; e <= 125 for finite fp32 input, so 127 - e is in [2, 254]),
// and below 8 because |v| < 2^(e + 3).
__device__ __forceinline__ float mx_scaled(uint32_t mag_bits, int e) {
    return __uint_as_float(mag_bits) * __uint_as_float((uint32_t)(127 - e) << 23);
}

// E2M1 code (sign clear) of r >= 0: round to nearest with the decision points at
// the midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5 and 5, where the even code wins;
// anything above 5 takes the largest magnitude, 6.  The code counts the decision
// points r has passed (strictly for those where the lower code is the even one),
// without branches, so the lanes of a warp never diverge.
__device__ __forceinline__ uint32_t e2m1_code(float r) {
    return (uint32_t)(r > 0.25f) + (uint32_t)(r >= 0.75f) + (uint32_t)(r > 1.25f) + (uint32_t)(r >= 1.75f) +
           (uint32_t)(r > 2.5f) + (uint32_t)(r >= 3.5f) + (uint32_t)(r > 5.0f);
}

// E2M1 codes (sign in bit 3) of two values already divided by their block scale
// (|v| < 8), packed as one byte with `lo` in the low nibble: the hardware
// conversion rounds to nearest with ties to the even code and saturates at 6, the
// rule e2m1_code implements with comparisons (a sign on a value that rounds to 0
// gives code 8).
__device__ __forceinline__ uint32_t e2m1_pair(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

}  // namespace moe

namespace moe {

// 2^k as a float, exactly, for k in [-149, 127] (subnormal below -126).
__device__ __forceinline__ float mx_pow2(int k) {
    return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(1u << (k + 149));
}

// Exponent of one term of an activation written as a sum of MXFP4 terms (the
// decode path, where the sum must reproduce the activation closely): the smallest
// e with max |v| <= 6 * 2^e, so no element saturates, clamped to [-127, 127].  For a
// normal max of 2^f * (1 + m) that is f - 2 when m <= 1/2, else f - 1; a subnormal
// max takes -127.
__device__ __forceinline__ int mx_term_exp(uint32_t amax_bits) {
    if ((amax_bits >> 23) == 0u) return -127;
    const int f = (int)(amax_bits >> 23) - 127;
    const int e = (amax_bits & 0x7fffffu) > 0x400000u ? f - 1 : f - 2;
    return max(-127, min(127, e));
}

// Value of E2M1 code c (sign bit 3) at block exponent e: twice the magnitudes
// {0, 0.5, 1, 1.5, 2, 3, 4, 6} are the nibbles of 0xC8643210.
__device__ __forceinline__ float mx_decode(uint32_t c, int e) {
    const float m = (float)((0xC8643210u >> (4 * (c & 7u))) & 0xFu) * mx_pow2(e - 1);
    return (c & 8u) ? -m : m;
}

}  // namespace moe
