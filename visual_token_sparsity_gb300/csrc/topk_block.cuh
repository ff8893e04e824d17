// Exact block-wide top-k of one row: the k largest scores, ties broken
// towards the lower index, written in ascending index order.
//
// Scores become order-preserving uint32 keys (-0.0 folded onto +0.0 so that
// float equality and key equality agree).  The row's smallest and largest
// keys fix the bits all keys share; MSB-first radix select then runs over the
// remaining bits in 8-bit windows (shared-memory histogram), narrowing a
// (prefix, mask) pair that brackets the k-th largest key, and stops as soon
// as the selected bin holds exactly the keys still needed (or every bit is
// fixed).  A block-wide scan over contiguous per-thread segments then emits
// keys above the prefix plus the lowest-index keys equal to it, in index
// order.
#pragma once

#include <stdint.h>

namespace sv {

struct TopkShared {
  int hist[256];
  int scan_tmp[33];
  uint32_t red_min[32], red_max[32];
  int sel_digit, sel_above, sel_count;
};

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t f = __float_as_uint(x);
  if (f == 0x80000000u) f = 0u;
  return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}

// Block-wide exclusive scan of one value per thread (blockDim.x a multiple
// of 32, at most 1024); unsigned types wrap modulo 2^32.
template <typename T>
__device__ __forceinline__ T block_exclusive_scan(T v, T* warp_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const T w = lane < nw ? warp_tmp[lane] : T(0);
    T wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const T t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < nw) warp_tmp[lane] = wi - w;
  }
  __syncthreads();
  const T res = warp_tmp[warp] + incl - v;
  __syncthreads();
  return res;
}

// Row `row`'s key count nr and selection size kr under per-sequence lengths
// (rows_per_seq rows per sequence; n and k are the capacities); (0, 0) when
// a length is out of range.
__device__ __forceinline__ void row_lengths(const SeqLens& lens, int row, int rows_per_seq, int n, int k,
                                            int& nr, int& kr) {
  SeqLens l = lens;
  l.n_text = nullptr;
  int nt;
  seq_lengths(l, row / rows_per_seq, n, 0, k, nr, nt, kr);
}

// Index slots [from, k) of a row that selected fewer than k tokens get -1
// (all threads of the block call this).
__device__ __forceinline__ void fill_unselected(int32_t* dst, int from, int k) {
  for (int i = from + (int)threadIdx.x; i < k; i += (int)blockDim.x) dst[i] = -1;
}

// All threads of the block call this.  keys: shared memory for n keys, or
// nullptr to re-read `src` (through L2) on every pass.  `src` may have been
// written by other CTAs of the running grid: it is read with ld.global.cg.
__device__ __forceinline__ void block_topk_row(const float* src, int n, int k, int32_t* dst,
                                               uint32_t* keys, TopkShared& ts) {
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  // stage the keys (four independent loads in flight per thread) and find
  // the smallest and largest key
  uint32_t lmin = 0xffffffffu, lmax = 0u;
  auto stage = [&](int i, float x) {
    const uint32_t key = order_key(x);
    if (keys) keys[i] = key;
    lmin = min(lmin, key);
    lmax = max(lmax, key);
  };
  int i0 = tid;
  if (keys != nullptr && (reinterpret_cast<uintptr_t>(src) & 15u) == 0) {
    // aligned row staged in shared memory: 16-byte loads, four per thread in
    // flight (a 2880-key row is one round of loads for 256 threads)
    const float4* s4 = reinterpret_cast<const float4*>(src);
    uint4* k4 = reinterpret_cast<uint4*>(keys);
    const int n4 = n >> 2;
    auto stage4 = [&](int v, float4 x) {
      const uint4 kk = make_uint4(order_key(x.x), order_key(x.y), order_key(x.z), order_key(x.w));
      k4[v] = kk;
      lmin = min(min(lmin, min(kk.x, kk.y)), min(kk.z, kk.w));
      lmax = max(max(lmax, max(kk.x, kk.y)), max(kk.z, kk.w));
    };
    int v = tid;
    for (; v + 3 * nt < n4; v += 4 * nt) {
      const float4 x0 = __ldcg(s4 + v), x1 = __ldcg(s4 + v + nt);
      const float4 x2 = __ldcg(s4 + v + 2 * nt), x3 = __ldcg(s4 + v + 3 * nt);
      stage4(v, x0);
      stage4(v + nt, x1);
      stage4(v + 2 * nt, x2);
      stage4(v + 3 * nt, x3);
    }
    for (; v < n4; v += nt) stage4(v, __ldcg(s4 + v));
    i0 = 4 * n4 + tid;
  } else {
    for (; i0 + 3 * nt < n; i0 += 4 * nt) {
      const float x0 = __ldcg(src + i0), x1 = __ldcg(src + i0 + nt);
      const float x2 = __ldcg(src + i0 + 2 * nt), x3 = __ldcg(src + i0 + 3 * nt);
      stage(i0, x0);
      stage(i0 + nt, x1);
      stage(i0 + 2 * nt, x2);
      stage(i0 + 3 * nt, x3);
    }
  }
  for (; i0 < n; i0 += nt) stage(i0, __ldcg(src + i0));
  for (int i = tid; i < 256; i += nt) ts.hist[i] = 0;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    lmin = min(lmin, __shfl_xor_sync(0xffffffffu, lmin, o));
    lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  }
  if (lane == 0) {
    ts.red_min[warp] = lmin;
    ts.red_max[warp] = lmax;
  }
  __syncthreads();
  uint32_t kmin = ts.red_min[0], kmax = ts.red_max[0];
  for (int w = 1; w < nw; ++w) {
    kmin = min(kmin, ts.red_min[w]);
    kmax = max(kmax, ts.red_max[w]);
  }
  auto key_at = [&](int i) -> uint32_t { return keys ? keys[i] : order_key(__ldcg(src + i)); };

  // (prefix, pmask): the known high bits of the k-th largest key; `remaining`
  // keys equal to it on those bits are still to be taken
  uint32_t prefix, pmask;
  int remaining = k;
  const uint32_t diff = kmin ^ kmax;
  if (diff == 0) {
    prefix = kmin;
    pmask = 0xffffffffu;
  } else {
    const int top = 31 - __clz(diff);               // highest bit where keys differ
    pmask = top == 31 ? 0u : ~((2u << top) - 1u);    // the bits above it are common
    prefix = kmin & pmask;
    int hi = top + 1;                                // next window: bits [lo, hi)
#pragma unroll 1
    while (hi > 0) {
      const int lo = hi > 8 ? hi - 8 : 0;
      const uint32_t wmask = (1u << (hi - lo)) - 1u;
      for (int i = tid; i < n; i += nt) {
        const uint32_t key = key_at(i);
        if ((key & pmask) == prefix) atomicAdd(&ts.hist[(key >> lo) & wmask], 1);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l scans bins 255-8l .. 248-8l (descending)
        int c[8], s = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          c[j] = ts.hist[255 - 8 * lane - j];
          s += c[j];
        }
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const int excl = incl - s;
        if (excl < remaining && remaining <= incl) {
          int run = excl;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (run + c[j] >= remaining) {
              ts.sel_digit = 255 - 8 * lane - j;
              ts.sel_above = run;
              ts.sel_count = c[j];
              break;
            }
            run += c[j];
          }
        }
      }
      __syncthreads();
      prefix |= (uint32_t)ts.sel_digit << lo;
      pmask |= wmask << lo;
      remaining -= ts.sel_above;
      const int cnt = ts.sel_count;
      __syncthreads();                       // every thread has read the selection
      if (cnt == remaining || lo == 0) break;  // the bin is taken whole, or the key is exact
      for (int i = tid; i < 256; i += nt) ts.hist[i] = 0;
      __syncthreads();
      hi = lo;
    }
  }

  // keys above the prefix are taken; of those equal to it, the `remaining`
  // lowest indices
  const int seg = (n + nt - 1) / nt;
  const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
  int gt = 0, eq = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t kp = key_at(i) & pmask;
    gt += kp > prefix;
    eq += kp == prefix;
  }
  int gt_before, eq_before;
  if (n < 65536) {   // both counts fit in 16 bits: one scan of the packed pair
    const uint32_t packed = block_exclusive_scan<uint32_t>(((uint32_t)gt << 16) | (uint32_t)eq,
                                                           reinterpret_cast<uint32_t*>(ts.scan_tmp));
    gt_before = (int)(packed >> 16);
    eq_before = (int)(packed & 0xffffu);
  } else {
    gt_before = block_exclusive_scan<int>(gt, ts.scan_tmp);
    eq_before = block_exclusive_scan<int>(eq, ts.scan_tmp);
  }
  int take_eq = remaining - eq_before;
  take_eq = take_eq < 0 ? 0 : (take_eq > eq ? eq : take_eq);
  int o = gt_before + min(eq_before, remaining);
  int e = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t kp = key_at(i) & pmask;
    bool take = kp > prefix;
    if (kp == prefix) {
      take = e < take_eq;
      ++e;
    }
    if (take) dst[o++] = i;
  }
}

}  // namespace sv
