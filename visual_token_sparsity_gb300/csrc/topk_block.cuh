// Exact block-wide top-k of one row: the k largest scores, ties broken
// towards the lower index, written in ascending index order.
//
// Scores become order-preserving uint32 keys (-0.0 folded onto +0.0 so that
// float equality and key equality agree).  A 4-pass MSB-first radix select
// (8-bit digits, shared-memory histogram) finds the exact k-th largest key T
// and how many keys equal to T are still needed; a block-wide scan over
// contiguous per-thread segments then emits the selection in index order,
// taking the equal-to-T keys with the lowest indices.
#pragma once

#include <stdint.h>

namespace sv {

struct TopkShared {
  int hist[256];
  int scan_tmp[33];
  int sel_digit, sel_above;
};

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t f = __float_as_uint(x);
  if (f == 0x80000000u) f = 0u;
  return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}

// Histogram increment aggregated over the lanes of a warp that hit the same
// bin (the leading digit of similar-magnitude floats falls into few bins, and
// same-address shared atomics serialise).  bin < 0 adds nothing.
__device__ __forceinline__ void hist_add(int* hist, int bin) {
  const unsigned peers = __match_any_sync(__activemask(), bin);
  if (bin >= 0 && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], __popc(peers));
}

// Block-wide exclusive scan of one int per thread (blockDim.x a multiple of
// 32, at most 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int w = lane < nw ? warp_tmp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < nw) warp_tmp[lane] = wi - w;
  }
  __syncthreads();
  const int res = warp_tmp[warp] + incl - v;
  __syncthreads();
  return res;
}

// All threads of the block call this.  keys: shared memory for n keys, or
// nullptr to re-read `src` (through L2) on every pass.  `src` may have been
// written by other CTAs of the running grid: it is read with ld.global.cg.
__device__ __forceinline__ void block_topk_row(const float* src, int n, int k, int32_t* dst,
                                               uint32_t* keys, TopkShared& ts) {
  const int tid = threadIdx.x, nt = blockDim.x;
  if (keys) {
    for (int i = tid; i < n; i += nt) keys[i] = order_key(__ldcg(src + i));
  }
  if (tid == 0) { ts.sel_digit = 0; ts.sel_above = 0; }
  __syncthreads();
  auto key_at = [&](int i) -> uint32_t { return keys ? keys[i] : order_key(__ldcg(src + i)); };

  uint32_t prefix = 0, pmask = 0;
  int remaining = k;
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += nt) ts.hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += nt) {
      const uint32_t key = key_at(i);
      hist_add(ts.hist, (key & pmask) == prefix ? (int)((key >> shift) & 255u) : -1);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l scans bins 255-8l .. 248-8l (descending)
      int c[8], s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = ts.hist[255 - 8 * tid - j]; s += c[j]; }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += t;
      }
      const int excl = incl - s;
      if (excl < remaining && remaining <= incl) {
        int run = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= remaining) { ts.sel_digit = 255 - 8 * tid - j; ts.sel_above = run; break; }
          run += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)ts.sel_digit << shift;
    pmask |= 255u << shift;
    remaining -= ts.sel_above;
    __syncthreads();
  }
  const uint32_t T = prefix;  // the exact k-th largest key; `remaining` keys equal to T are taken

  const int seg = (n + nt - 1) / nt;
  const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
  int gt = 0, eq = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t key = key_at(i);
    gt += key > T;
    eq += key == T;
  }
  const int eq_before = block_exclusive_scan(eq, ts.scan_tmp);
  int take_eq = remaining - eq_before;
  take_eq = take_eq < 0 ? 0 : (take_eq > eq ? eq : take_eq);
  int o = block_exclusive_scan(gt + take_eq, ts.scan_tmp);
  int e = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t key = key_at(i);
    bool take = key > T;
    if (key == T) { take = e < take_eq; ++e; }
    if (take) dst[o++] = i;
  }
}

}  // namespace sv
