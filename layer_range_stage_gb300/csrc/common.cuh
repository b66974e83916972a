// Device helpers shared by the stage kernels (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lrs {

constexpr int kWarp = 32;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// 16 weight bytes, read once: streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ld_stream_u4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const void* p) {
  uint16_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

// Exact int8 -> float for the 4 bytes of a word.  The byte is biased by 128 (xor 0x80),
// placed as the low mantissa byte of 2^23 (exponent byte 0x4B) with one byte permute,
// and the bias 2^23 + 128 is subtracted: 2^23 + (q + 128) - (2^23 + 128) = q, exactly.
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float& a, float& b, float& c, float& d) {
  const uint32_t x = w ^ 0x80808080u;
  const float bias = 8388736.0f;
  a = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540)) - bias;
  b = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7541)) - bias;
  c = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7542)) - bias;
  d = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7543)) - bias;
}

// sum_j q_j * x_j over the 16 int8 weights of w and 16 floats of x.
__device__ __forceinline__ float dot16_i8(const uint4 w, const float4 x0, const float4 x1, const float4 x2,
                                          const float4 x3) {
  float a, b, c, d, acc;
  i8x4_to_f32(w.x, a, b, c, d);
  acc = a * x0.x;
  acc = fmaf(b, x0.y, acc);
  acc = fmaf(c, x0.z, acc);
  acc = fmaf(d, x0.w, acc);
  i8x4_to_f32(w.y, a, b, c, d);
  acc = fmaf(a, x1.x, acc);
  acc = fmaf(b, x1.y, acc);
  acc = fmaf(c, x1.z, acc);
  acc = fmaf(d, x1.w, acc);
  i8x4_to_f32(w.z, a, b, c, d);
  acc = fmaf(a, x2.x, acc);
  acc = fmaf(b, x2.y, acc);
  acc = fmaf(c, x2.z, acc);
  acc = fmaf(d, x2.w, acc);
  i8x4_to_f32(w.w, a, b, c, d);
  acc = fmaf(a, x3.x, acc);
  acc = fmaf(b, x3.y, acc);
  acc = fmaf(c, x3.z, acc);
  acc = fmaf(d, x3.w, acc);
  return acc;
}

__device__ __forceinline__ float h2f_bits(uint16_t h) { return __half2float(__ushort_as_half(h)); }

__device__ __forceinline__ float silu(float z) { return z / (1.0f + expf(-z)); }

}  // namespace lrs
