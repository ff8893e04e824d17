// Packed fp32x2 arithmetic and an FMA-pipe exp2 for the salience softmax.
//
// sm_100-family parts execute fma/add/mul on fp32 pairs ("f32x2") in one
// instruction, which halves the issue cost of the element-wise softmax work.
// exp2 normally runs on the MUFU unit (16 results per clock per SM), the
// bottleneck of the salience kernel; exp2_poly2 computes it on the FMA pipe
// instead so a fraction of the elements can bypass MUFU:
//   x is clamped to [-126, 0]; adding the shifter 1.5 * 2^23 rounds x to the
//   nearest integer j in the low mantissa bits (range reduction as in
//   Cody & Waite, "Software Manual for the Elementary Functions", 1980);
//   f = x - j lies in [-1/2, 1/2]; 2^f is a degree-4 polynomial whose
//   coefficients are this library's own minimax (Remez exchange) fit for
//   relative error on [-1/2, 1/2] (max 2.6e-6; 2.7e-6 evaluated in fp32);
//   2^j is applied by adding j to the exponent field: the shifter's bit
//   pattern shifted left by 23 wraps to exactly j << 23 (mod 2^32).
#pragma once

#include <stdint.h>

namespace sv {
namespace fm {

// Remez fit of 2^f on [-1/2, 1/2], p(f) = c0 + c1 f + c2 f^2 + c3 f^3 + c4 f^4.
constexpr float kExp2C0 = 0.9999992847442627f;
constexpr float kExp2C1 = 0.6931217908859253f;
constexpr float kExp2C2 = 0.240247443318367f;
constexpr float kExp2C3 = 0.05591785907745361f;
constexpr float kExp2C4 = 0.009570102207362652f;
constexpr float kShifter = 12582912.0f;  // 1.5 * 2^23
constexpr float kExp2Min = -126.0f;

__device__ __forceinline__ uint64_t pack2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t splat2(float a) { return pack2(a, a); }
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float ex2_mufu(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint64_t exp2_mufu2(uint64_t x) {
  float a, b;
  unpack2(x, a, b);
  return pack2(ex2_mufu(a), ex2_mufu(b));
}

// 2^x for a pair, on the FMA pipe; inputs below -126 (and -inf) give 2^-126.
__device__ __forceinline__ uint64_t exp2_poly2(uint64_t x) {
  float a, b;
  unpack2(x, a, b);
  const uint64_t xc = pack2(fmaxf(a, kExp2Min), fmaxf(b, kExp2Min));
  const uint64_t t = add2(xc, splat2(kShifter));
  const uint64_t j = add2(t, splat2(-kShifter));
  const uint64_t f = fma2(j, splat2(-1.0f), xc);
  uint64_t p = fma2(splat2(kExp2C4), f, splat2(kExp2C3));
  p = fma2(p, f, splat2(kExp2C2));
  p = fma2(p, f, splat2(kExp2C1));
  p = fma2(p, f, splat2(kExp2C0));
  float p0, p1, t0, t1;
  unpack2(p, p0, p1);
  unpack2(t, t0, t1);
  const uint32_t r0 = __float_as_uint(p0) + (__float_as_uint(t0) << 23);
  const uint32_t r1 = __float_as_uint(p1) + (__float_as_uint(t1) << 23);
  return pack2(__uint_as_float(r0), __uint_as_float(r1));
}

}  // namespace fm
}  // namespace sv
