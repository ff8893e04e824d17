// Row-wise exact top-k with lowest-index tie-break and ascending output.
//
// The selection step of both SparseVILA phases (velog.io summary §3.1: prune
// the lowest-salience tokens; §3.2: keep the highest-scoring cached tokens
// active; xllm-io review §五 topk).
//
// One CTA per row.  Scores are mapped to order-preserving uint32 keys (with
// -0.0 folded onto +0.0 so that float equality and key equality agree) and
// staged in shared memory when the row fits.  A 4-pass MSB-first radix select
// (8-bit digits, shared-memory histograms) finds the exact k-th largest key T
// and how many keys equal to T are still needed; a block-wide scan over
// contiguous per-thread segments then emits the selected indices in ascending
// order, taking the equal-to-T keys with the lowest indices.
#include "common.cuh"
#include "kernels.h"

namespace sv {

__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t f = __float_as_uint(x);
  if (f == 0x80000000u) f = 0u;
  return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}

// Block-wide exclusive scan of one int per thread (blockDim.x multiple of 32,
// <= 1024).  Returns the exclusive prefix; *total gets the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tmp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nw ? warp_tmp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    if (lane < nw) warp_tmp[lane] = wi - w;
    if (lane == 31) warp_tmp[32] = wi;
  }
  __syncthreads();
  int res = warp_tmp[warp] + incl - v;
  *total = warp_tmp[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(1024)
topk_rows_kernel(const float* __restrict__ scores, int n, int k, int32_t* __restrict__ idx,
                 int keys_in_smem) {
  extern __shared__ uint32_t smem_keys[];
  __shared__ int hist[256];
  __shared__ int scan_tmp[33];
  __shared__ int sel_digit, sel_above;

  const int row = blockIdx.x;
  const float* src = scores + (size_t)row * n;
  const int tid = threadIdx.x;
  const int nt = blockDim.x;

  if (keys_in_smem) {
    for (int i = tid; i < n; i += nt) smem_keys[i] = order_key(__ldg(src + i));
  }
  __syncthreads();

  uint32_t prefix = 0, pmask = 0;
  int remaining = k;
  if (tid == 0) { sel_digit = 0; sel_above = 0; }
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    for (int i = tid; i < 256; i += nt) hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < n; i += nt) {
      const uint32_t key = keys_in_smem ? smem_keys[i] : order_key(__ldg(src + i));
      if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 32) {
      // lane l scans bins 255-8l .. 248-8l (descending)
      int c[8], s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = hist[255 - 8 * tid - j]; s += c[j]; }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += t;
      }
      const int excl = incl - s;
      if (excl < remaining && remaining <= incl) {
        int run = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (run + c[j] >= remaining) { sel_digit = 255 - 8 * tid - j; sel_above = run; break; }
          run += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sel_digit << shift;
    pmask |= 255u << shift;
    remaining -= sel_above;
    __syncthreads();
  }
  const uint32_t T = prefix;  // exact k-th largest key; `remaining` keys equal to T are taken

  // contiguous segment per thread
  const int seg = (n + nt - 1) / nt;
  const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
  int gt = 0, eq = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t key = keys_in_smem ? smem_keys[i] : order_key(__ldg(src + i));
    gt += key > T;
    eq += key == T;
  }
  int total;
  const int eq_before = block_exclusive_scan(eq, scan_tmp, &total);
  int take_eq = remaining - eq_before;
  take_eq = take_eq < 0 ? 0 : (take_eq > eq ? eq : take_eq);
  const int out_pos = block_exclusive_scan(gt + take_eq, scan_tmp, &total);
  int32_t* dst = idx + (size_t)row * k;
  int o = out_pos, e = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t key = keys_in_smem ? smem_keys[i] : order_key(__ldg(src + i));
    bool take = key > T;
    if (key == T) { take = e < take_eq; ++e; }
    if (take) dst[o++] = i;
  }
}

int topk_max_smem_keys() { return 52 * 1024; }   // 208 KB of keys

cudaError_t launch_topk_rows(const float* scores, int rows, int n, int k, int32_t* idx,
                             cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const bool in_smem = n <= topk_max_smem_keys();
  const size_t smem = in_smem ? (size_t)n * sizeof(uint32_t) : 0;
  int threads = n >= 16384 ? 1024 : (n >= 2048 ? 512 : 256);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(topk_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             topk_max_smem_keys() * (int)sizeof(uint32_t));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  topk_rows_kernel<<<rows, threads, smem, stream>>>(scores, n, k, idx, in_smem ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace sv
