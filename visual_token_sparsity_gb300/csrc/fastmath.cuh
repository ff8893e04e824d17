// Packed fp32x2 arithmetic for the salience softmax.
//
// sm_100-family parts execute fma/add/mul on fp32 pairs ("f32x2") in one
// instruction, which halves the issue cost of the element-wise softmax work.
// exp2 runs on the MUFU unit: ex2.approx.ftz.f32 sustains 32 results per clock
// per SM on GB300 (measured; the packed f16x2 / bf16x2 forms give the same 32
// per clock, so they would save issue slots but not exp throughput, and their
// 16-bit inputs are too coarse for softmax arguments).
#pragma once

#include <stdint.h>

namespace sv {
namespace fm {

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
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
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

}  // namespace fm
}  // namespace sv
