// The dequant-fused dot product shared by the decode GEMV and the persistent decode
// kernel.
//
// Weights are stored biased, b = q + 128 in [1, 255] (one byte per weight), with one fp16
// scale per block of 32 along K.  For 16 weights w_j = s * (b_j - 128) and inputs x_j:
//   sum_j w_j x_j = s * (sum_j b_j x_j - 128 * X),   X = sum_j x_j (per 16-input chunk).
// b_j is turned into a float without any arithmetic: the byte moved into an otherwise
// zero word is the denormal b_j * 2^-149, exactly.  With inputs pre-scaled by 2^64 the
// products b_j * x_j * 2^-85 are normal floats for |x_j| >= 2^-41, so one FFMA per weight
// accumulates them (IEEE denormal operands, no flush-to-zero); the chunk sum is rescaled by
// 2^85 (exact) and corrected by -128 X in one FFMA, then multiplied by the block scale.
// Smaller inputs give denormal products, off by at most 2^-65 s each after the rescale; inputs
// must stay below 2^64 in magnitude (the scaled input overflows there).  The error is float32
// rounding measured against the biased magnitudes, sum_j b_j |x_j| + 128 |X|.
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
// D_i as a float.  Beyond float32 accumulation the roundings are those of N_j, rint of the
// float32 product h_j * (1/u) (at most u / 2 + 2^-24 |h_j| per input: below 1.51 * 2^-23 of the
// chunk's largest input, where float32 keeps 2^-24), and of u itself (relative 2^-24, the same
// for the whole chunk).
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23

__device__ __forceinline__ int dp4a_us(unsigned a, unsigned b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// The chunk form of 16 inputs: limbs l0, l1, l2 (byte j of word j / 4 is input j's) and
// k = (the three dp4a starting values, bits of u), computed by two adjacent lanes
// (half = lane & 1), each holding inputs 8 half .. 8 half + 7 of the chunk in h: words 2 half
// and 2 half + 1 of l0, l1, l2 and of k come back in (lw0, lw1, lw2, kw).  Both lanes must
// call it together.  The three limbs of N_j are the bytes of N_j + 0x808080 (each limb plus
// 128: a base-256 representation with digits in [0, 255], and below 2^24 since
// |N_j| < 2^23), so they are picked out by byte permutes and their bias removed by one XOR per
// word; the limb sums are dp4a against ones.
__device__ __forceinline__ void q8_chunk_encode2(const float h[8], int half, uint2& lw0, uint2& lw1, uint2& lw2,
                                                 uint2& kw) {
  float m = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(h[j]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  const int e = max((int)((__float_as_uint(m) >> 23) & 0xFFu) - 126, -100);
  const float sc = __int_as_float((unsigned)(127 + 23 - e) << 23) * 0.9921875f;
  unsigned w[3][2];
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    unsigned v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = (unsigned)(__float2int_rn(h[4 * q + j] * sc) + 0x808080);
    const unsigned ablo = __byte_perm(v[0], v[1], 0x5140), abhi = __byte_perm(v[0], v[1], 0x7362);
    const unsigned cdlo = __byte_perm(v[2], v[3], 0x5140), cdhi = __byte_perm(v[2], v[3], 0x7362);
    w[0][q] = __byte_perm(abhi, cdhi, 0x5410) ^ 0x80808080u;  // byte 2: l0
    w[1][q] = __byte_perm(ablo, cdlo, 0x7632) ^ 0x80808080u;  // byte 1: l1
    w[2][q] = __byte_perm(ablo, cdlo, 0x5410) ^ 0x80808080u;  // byte 0: l2
  }
  int s[3];
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    s[i] = __dp4a((int)w[i][1], 0x01010101, __dp4a((int)w[i][0], 0x01010101, 0));
    s[i] += __shfl_xor_sync(0xffffffffu, s[i], 1);
  }
  lw0 = make_uint2(w[0][0], w[0][1]);
  lw1 = make_uint2(w[1][0], w[1][1]);
  lw2 = make_uint2(w[2][0], w[2][1]);
  const unsigned unit = __float_as_uint(__int_as_float((unsigned)(127 + e - 23) << 23) * (128.0f / 127.0f));
  kw = half ? make_uint2((unsigned)(0x4B400000 - 128 * s[2]), unit)
            : make_uint2((unsigned)(0x4B400000 - 128 * s[0]), (unsigned)(0x4B400000 - 128 * s[1]));
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
