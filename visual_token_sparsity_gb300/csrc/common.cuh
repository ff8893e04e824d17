// Device helpers shared by the libsv kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

constexpr int kBlockTokens = 16;
constexpr int kStatusBadBlock = 0x1;
constexpr int kStatusBadIndex = 0x2;
constexpr int kStatusTimeout = 0x10;   // a bounded wait inside a kernel gave up
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void flag_status(int* status, int bits) { atomicOr(status, bits); }

// Two bf16 values packed in a 32-bit word -> fp32 (exact).
__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// fp32 -> bf16 bits, round to nearest even (finite inputs).
__device__ __forceinline__ uint32_t f32_to_bf16_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7f800000u) == 0x7f800000u) return (u >> 16) | ((u & 0xffffu) ? 0x40u : 0u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

// 16-byte streaming load through the non-coherent path, not kept in L1,
// with a 256-byte L2 prefetch hint.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Butterfly reduce-scatter of NV per-lane partial sums over aligned groups of
// LPT lanes.  Afterwards every lane holds the full group sum of value index
// (lane % LPT) / (LPT / NV); LPT / NV lanes hold each value.
template <int NV, int LPT, int M = LPT / 2>
struct GroupReduce {
  static __device__ __forceinline__ void run(float* v, int lane) {
    if constexpr (M >= 1) {
      if constexpr (NV > 1) {
        constexpr int H = NV / 2;
        const bool upper = (lane & M) != 0;
#pragma unroll
        for (int i = 0; i < H; ++i) {
          float send = upper ? v[i] : v[i + H];
          float keep = upper ? v[i + H] : v[i];
          v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
        }
        GroupReduce<H, LPT, M / 2>::run(v, lane);
      } else {
        v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
        GroupReduce<1, LPT, M / 2>::run(v, lane);
      }
    }
  }
};

}  // namespace sv
