// Packed fp32 pairs (sm_100 f32x2 arithmetic; both halves rounded to nearest
// even, like the scalar __fmul_rn / __fadd_rn / __fmaf_rn).
//
// ptxas fuses a packed multiply into a following packed add even with .rn
// (measured: a product of exactly 6.5 followed by + 1.5 * 2^23 rounded as if
// fused), so a packed add must never consume a packed product directly where
// the separate rounding matters.
#pragma once

#include <cstdint>

namespace awq {

typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pack2(float a, float b) {
  return static_cast<f32x2>(__float_as_uint(a)) | (static_cast<f32x2>(__float_as_uint(b)) << 32);
}
__device__ __forceinline__ float lo2(f32x2 v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi2(f32x2 v) {
  return __uint_as_float(static_cast<uint32_t>(v >> 32));
}
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

}  // namespace awq
