// Device helpers shared by the libsv kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

namespace sv {

constexpr int kBlockTokens = 16;
constexpr int kStatusBadBlock = 0x1;
constexpr int kStatusBadIndex = 0x2;
constexpr int kStatusBadLength = 0x4;  // a per-sequence length outside its capacity
constexpr int kStatusTimeout = 0x10;   // a bounded wait inside a kernel gave up
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void flag_status(int* status, int bits) { atomicOr(status, bits); }

// Programmatic dependent launch.  A kernel launched by launch_dependent()
// may become resident while the kernel before it in the stream drains; it
// calls grid_dep_sync() first thing, which waits until that kernel has
// completed and its memory operations are visible, and then lets its own
// successor launch early.  Both are no-ops in an ordinary launch.
__device__ __forceinline__ void grid_dep_sync() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kernel` with programmatic stream serialisation (overlapping its
// launch and CTA rasterisation with the previous kernel's tail) unless the
// environment sets SV_PDL=0.
bool pdl_enabled();
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Sequence b's visual, text and selected counts under `s`, whose capacities
// are n_vis, n_text and k.  False (counts set to 0) when a count lies outside
// [0, its capacity] or the selection exceeds the visual count: the caller
// skips the sequence and reports kStatusBadLength.
__device__ __forceinline__ bool seq_lengths(const SeqLens& s, int b, int n_vis, int n_text, int k,
                                            int& nv, int& nt, int& kb) {
  nv = s.n_vis ? __ldg(s.n_vis + b) : n_vis;
  nt = s.n_text ? __ldg(s.n_text + b) : n_text;
  kb = s.k ? __ldg(s.k + b) : k;
  if (nv < 0 || nv > n_vis || nt < 0 || nt > n_text || kb < 0 || kb > k || kb > nv) {
    nv = nt = kb = 0;
    return false;
  }
  return true;
}

// Attention token counts of sequence b: visual nv, text nt and attended
// visual kb (the k_vis listed indices, or all nv visual tokens when there is
// no index list).  Out-of-range lengths attend nothing; `report` selects the
// one thread that sets kStatusBadLength.
__device__ __forceinline__ bool attn_lengths(const SeqLens& lens, bool indexed, int b, int n_vis,
                                             int n_text, int k_vis, bool report, int* status, int& nv,
                                             int& nt, int& kb) {
  nv = n_vis;
  nt = n_text;
  kb = indexed ? k_vis : n_vis;
  if (!lens.any()) return true;
  SeqLens l = lens;
  if (!indexed) l.k = nullptr;
  const bool ok = seq_lengths(l, b, n_vis, n_text, indexed ? k_vis : 0, nv, nt, kb);
  if (!indexed) kb = nv;
  if (!ok && report) flag_status(status, kStatusBadLength);
  return ok;
}

// Row id (page * Hkv + g) * 16 + slot of the cache position `pos` of KV head
// g, or kNoRowId (kStatusBadBlock) when the page id is outside the pool.
constexpr uint32_t kNoRowId = 0xffffffffu;
// The token a fused append-and-attend call appends: read from the caller's
// k_new / v_new instead of the pool (a pool row id is at most 2^32 - 17).
constexpr uint32_t kNewRowId = 0xfffffffeu;

// One warp stores the appended token's K and V rows (bf16 [d] each, from
// k_new / v_new of (sequence b, KV head g)) at cache position pos; a page id
// outside the pool is reported and skipped, as by the append kernel.
__device__ __forceinline__ void store_new_token(uint16_t* k_pool, uint16_t* v_pool, const uint16_t* k_new,
                                                const uint16_t* v_new, const int32_t* bt, int num_blocks,
                                                int Hkv, int D, int b, int g, int pos, int lane) {
  const int page = __ldg(bt + (pos >> 4));
  if (page < 0 || page >= num_blocks) return;   // reported by the attention's row lookup
  const size_t row = ((size_t)page * Hkv + g) * 16 + (pos & 15);
  const size_t src = ((size_t)b * Hkv + g) * D;
  const int cpr = D / 8;                          // 16-byte words per row
  for (int v = lane; v < 2 * cpr; v += 32) {
    const bool is_k = v < cpr;
    const int c = is_k ? v : v - cpr;
    const uint4 x = *reinterpret_cast<const uint4*>((is_k ? k_new : v_new) + src + c * 8);
    *reinterpret_cast<uint4*>((is_k ? k_pool : v_pool) + row * D + c * 8) = x;
  }
}

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

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte asynchronous copy global -> shared, cached in L2 only; src_bytes 0
// writes 16 zero bytes (no global read)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

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
