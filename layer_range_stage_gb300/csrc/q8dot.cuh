// The dequant-fused dot product shared by the decode GEMV and the persistent decode
// kernel.
//
// Weights are stored biased, b = q + 128 in [1, 255] (one byte per weight), with one fp16
// scale per block of 32 along K.  For 16 weights w_j = s * (b_j - 128) and inputs x_j:
//   sum_j w_j x_j = s * (sum_j b_j x_j - 128 * X),   X = sum_j x_j (per 16-input chunk).
// b_j is turned into a float without any arithmetic: the byte moved into an otherwise
// zero word is the denormal b_j * 2^-149, exactly.  With inputs pre-scaled by 2^64 the
// products b_j * x_j * 2^-85 are normal floats, so one FFMA per weight accumulates them
// (IEEE denormal operands, no flush-to-zero); the chunk sum is rescaled by 2^85 (exact) and
// corrected by -128 X in one FFMA, then multiplied by the block scale.
#pragma once

#include <stdint.h>

namespace lrs {

constexpr float kXScale = 18446744073709551616.0f;        // 2^64
constexpr float kPScale = 38685626227668133590597632.0f;  // 2^85

// Byte j of a word as the denormal b_j * 2^-149 (one instruction each).
__device__ __forceinline__ float q8_b0(unsigned w) { return __uint_as_float(w & 0xFFu); }
__device__ __forceinline__ float q8_b1(unsigned w) { return __uint_as_float(__byte_perm(w, 0u, 0x4441)); }
__device__ __forceinline__ float q8_b2(unsigned w) { return __uint_as_float(__byte_perm(w, 0u, 0x4442)); }
__device__ __forceinline__ float q8_b3(unsigned w) { return __uint_as_float(w >> 24); }

// sum_j b_j * x'_j * 2^-149 over the 16 biased weight bytes of w (see above).
__device__ __forceinline__ float dot16_u8(const uint4 w, const float4 x0, const float4 x1, const float4 x2,
                                          const float4 x3) {
  float acc = __uint_as_float(w.x & 0xFFu) * x0.x;
  acc = fmaf(__uint_as_float(__byte_perm(w.x, 0u, 0x4441)), x0.y, acc);
  acc = fmaf(__uint_as_float(__byte_perm(w.x, 0u, 0x4442)), x0.z, acc);
  acc = fmaf(__uint_as_float(w.x >> 24), x0.w, acc);
  acc = fmaf(__uint_as_float(w.y & 0xFFu), x1.x, acc);
  acc = fmaf(__uint_as_float(__byte_perm(w.y, 0u, 0x4441)), x1.y, acc);
  acc = fmaf(__uint_as_float(__byte_perm(w.y, 0u, 0x4442)), x1.z, acc);
  acc = fmaf(__uint_as_float(w.y >> 24), x1.w, acc);
  acc = fmaf(__uint_as_float(w.z & 0xFFu), x2.x, acc);
  acc = fmaf(__uint_as_float(__byte_perm(w.z, 0u, 0x4441)), x2.y, acc);
  acc = fmaf(__uint_as_float(__byte_perm(w.z, 0u, 0x4442)), x2.z, acc);
  acc = fmaf(__uint_as_float(w.z >> 24), x2.w, acc);
  acc = fmaf(__uint_as_float(w.w & 0xFFu), x3.x, acc);
  acc = fmaf(__uint_as_float(__byte_perm(w.w, 0u, 0x4441)), x3.y, acc);
  acc = fmaf(__uint_as_float(__byte_perm(w.w, 0u, 0x4442)), x3.z, acc);
  acc = fmaf(__uint_as_float(w.w >> 24), x3.w, acc);
  return acc;
}

}  // namespace lrs
