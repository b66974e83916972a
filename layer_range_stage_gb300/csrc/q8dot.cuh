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

// ---- integer form of the staged input (the persistent decode)
//
// A chunk of 16 inputs h_j becomes an exponent e (every |h_j| < 2^e) and integers
// N_j = rint(h_j / u), u = (128/127) 2^(e - 23), so |N_j| < (127/128) 2^23 and each N_j is three
// signed bytes N_j = l0_j 2^16 + l1_j 2^8 + l2_j (l0_j within [-127, 127] even after the
// borrows of the lower bytes).  For 16 biased weight bytes b_j = q_j + 128:
//   sum_j q_j h_j = u (2^16 D0 + 2^8 D1 + D2) + (the rounding of the N_j),
//   D_i = sum_j b_j li_j - 128 sum_j li_j,
// each D_i an exact integer (|D_i| < 2^19) from four dp4a instructions on the weight words as
// they are: no weight is converted.  Starting a dp4a chain at 0x4B400000 - 128 sum_j li_j makes
// its result the float bits of 1.5 * 2^23 + D_i (exact while |D_i| < 2^22), so one FADD recovers
// D_i as a float.  Beyond float32 accumulation the roundings are those of N_j (at most u / 2 per
// input: relative 2^-23 of the chunk's largest input, where float32 keeps 2^-24) and of u
// itself (relative 2^-24, the same for the whole chunk).
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

__device__ __forceinline__ int dp4a_us(unsigned a, unsigned b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The limbs (l0, l1, l2: byte j of word j / 4 is input j's) and k = (the three dp4a starting
// values, bits of u) of a chunk of 16 inputs.
__device__ __forceinline__ void q8_chunk_encode(const float h[16], uint4& l0, uint4& l1, uint4& l2, uint4& k) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) m = fmaxf(m, fabsf(h[j]));
  // m = f 2^e with f in [0.5, 1); chunks below 2^-100 keep e = -100 (their integers are 0)
  const int e = max((int)((__float_as_uint(m) >> 23) & 0xFFu) - 126, -100);
  const float sc = __int_as_float((unsigned)(127 + 23 - e) << 23) * 0.9921875f;  // 1 / u = (127/128) 2^(23 - e)
  unsigned w0[4] = {0u, 0u, 0u, 0u}, w1[4] = {0u, 0u, 0u, 0u}, w2[4] = {0u, 0u, 0u, 0u};
  int s0 = 0, s1 = 0, s2 = 0;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int n = __float2int_rn(h[j] * sc);
    const int b2 = ((n + 128) & 255) - 128;
    const int n1 = (n - b2) >> 8;
    const int b1 = ((n1 + 128) & 255) - 128;
    const int b0 = (n1 - b1) >> 8;
    s0 += b0;
    s1 += b1;
    s2 += b2;
    w0[j >> 2] |= ((unsigned)b0 & 0xFFu) << (8 * (j & 3));
    w1[j >> 2] |= ((unsigned)b1 & 0xFFu) << (8 * (j & 3));
    w2[j >> 2] |= ((unsigned)b2 & 0xFFu) << (8 * (j & 3));
  }
  l0 = make_uint4(w0[0], w0[1], w0[2], w0[3]);
  l1 = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  l2 = make_uint4(w2[0], w2[1], w2[2], w2[3]);
  k = make_uint4((unsigned)(0x4B400000 - 128 * s0), (unsigned)(0x4B400000 - 128 * s1),
                 (unsigned)(0x4B400000 - 128 * s2),
                 __float_as_uint(__int_as_float((unsigned)(127 + e - 23) << 23) * (128.0f / 127.0f)));
}

// 2^16 D0 + 2^8 D1 + D2 (see above) for the 16 biased weight bytes of w.
__device__ __forceinline__ float q8_chunk_dot(const uint4 w, const uint4 l0, const uint4 l1, const uint4 l2,
                                              const uint4 k) {
  int r0 = (int)k.x, r1 = (int)k.y, r2 = (int)k.z;
  r0 = dp4a_us(w.x, l0.x, r0);
  r1 = dp4a_us(w.x, l1.x, r1);
  r2 = dp4a_us(w.x, l2.x, r2);
  r0 = dp4a_us(w.y, l0.y, r0);
  r1 = dp4a_us(w.y, l1.y, r1);
  r2 = dp4a_us(w.y, l2.y, r2);
  r0 = dp4a_us(w.z, l0.z, r0);
  r1 = dp4a_us(w.z, l1.z, r1);
  r2 = dp4a_us(w.z, l2.z, r2);
  r0 = dp4a_us(w.w, l0.w, r0);
  r1 = dp4a_us(w.w, l1.w, r1);
  r2 = dp4a_us(w.w, l2.w, r2);
  const float f0 = __int_as_float(r0) - kMagic, f1 = __int_as_float(r1) - kMagic, f2 = __int_as_float(r2) - kMagic;
  return fmaf(f0, 65536.0f, fmaf(f1, 256.0f, f2));
}

}  // namespace lrs
