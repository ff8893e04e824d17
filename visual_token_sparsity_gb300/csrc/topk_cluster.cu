// Row top-k for long rows on a thread-block cluster.
//
// The selection step of decode retrieval (velog.io SparseVILA summary §3.2)
// for long-video caches, where one (sequence, KV head) row holds tens of
// thousands of visual scores and a batch has only a few rows.  A cluster of
// kTopkClusterCtas CTAs owns one row; CTA r keeps the r-th slice of the row's
// order-preserving keys in its shared memory.  Each of the four radix passes
// builds a local 256-bin histogram, and after a cluster barrier every CTA
// sums the cluster's histograms through distributed shared memory and picks
// the same digit (histograms are double-buffered, so one cluster barrier per
// pass is enough).  The output phase exchanges per-CTA (greater, equal) counts
// the same way, so the CTAs write disjoint ranges of the ascending index list,
// with ties broken towards the lower index exactly as in the single-CTA
// routine (topk_block.cuh).  The cluster barriers are hardware barriers over
// co-scheduled CTAs; nothing spins.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"
#include "topk_block.cuh"

namespace cg = cooperative_groups;

namespace sv {

namespace {
constexpr int kTopkClusterCtas = 8;
constexpr int kTopkClusterThreads = 512;
}  // namespace

__global__ void __cluster_dims__(kTopkClusterCtas, 1, 1) __launch_bounds__(kTopkClusterThreads)
topk_cluster_kernel(const float* __restrict__ scores, int n, int k, int32_t* __restrict__ idx) {
  extern __shared__ uint32_t keys[];
  __shared__ int hist[2][256];    // double-buffered: peers read pass p's while pass p+1 fills the other
  __shared__ int total[256];
  __shared__ int scan_tmp[33];
  __shared__ int sel_digit, sel_above;
  __shared__ int cnt[2];          // this CTA's (greater, equal) counts
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.y;
  const int tid = threadIdx.x, nt = blockDim.x;
  const int slice = (n + kTopkClusterCtas - 1) / kTopkClusterCtas;
  const int lo = min(n, rank * slice), hi = min(n, lo + slice);
  const int m = hi - lo;
  const float* src = scores + (size_t)row * n + lo;
  for (int i = tid; i < m; i += nt) keys[i] = order_key(__ldcg(src + i));

  uint32_t prefix = 0, pmask = 0;
  int remaining = k;
  if (tid == 0) { sel_digit = 0; sel_above = 0; }
#pragma unroll 1
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    int* hcur = hist[pass & 1];
    for (int i = tid; i < 256; i += nt) hcur[i] = 0;
    __syncthreads();
    for (int i = tid; i < m; i += nt) {
      const uint32_t key = keys[i];
      hist_add(hcur, (key & pmask) == prefix ? (int)((key >> shift) & 255u) : -1);
    }
    cluster.sync();                                   // all local histograms complete
    for (int b = tid; b < 256; b += nt) {
      int s = 0;
#pragma unroll
      for (int r = 0; r < kTopkClusterCtas; ++r) s += cluster.map_shared_rank(hcur, r)[b];
      total[b] = s;
    }
    __syncthreads();
    if (tid < 32) {
      int c[8], s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = total[255 - 8 * tid - j]; s += c[j]; }
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
          if (run + c[j] >= remaining) { sel_digit = 255 - 8 * tid - j; sel_above = run; break; }
          run += c[j];
        }
      }
    }
    __syncthreads();
    prefix |= (uint32_t)sel_digit << shift;
    pmask |= 255u << shift;
    remaining -= sel_above;
    __syncthreads();          // total / sel_* are rewritten by the next pass
  }
  const uint32_t T = prefix;

  // this CTA's counts, then the counts of the CTAs before it in the row
  const int seg = (m + nt - 1) / nt;
  const int s0 = min(m, tid * seg), s1 = min(m, s0 + seg);
  int gt = 0, eq = 0;
  for (int i = s0; i < s1; ++i) {
    gt += keys[i] > T;
    eq += keys[i] == T;
  }
  if (tid == 0) cnt[0] = cnt[1] = 0;
  __syncthreads();
  int w_gt = gt, w_eq = eq;
#pragma unroll
  for (int o2 = 16; o2 >= 1; o2 >>= 1) {
    w_gt += __shfl_xor_sync(0xffffffffu, w_gt, o2);
    w_eq += __shfl_xor_sync(0xffffffffu, w_eq, o2);
  }
  if ((tid & 31) == 0) { atomicAdd(&cnt[0], w_gt); atomicAdd(&cnt[1], w_eq); }
  cluster.sync();
  int gt_before = 0, eq_before_cta = 0;
  for (int r = 0; r < rank; ++r) {
    const int* rc = cluster.map_shared_rank(cnt, r);
    gt_before += rc[0];
    eq_before_cta += rc[1];
  }
  const int take_before = min(eq_before_cta, remaining);   // equal keys taken by earlier CTAs
  const int eq_before = block_exclusive_scan(eq, scan_tmp) + eq_before_cta;
  int take_eq = remaining - eq_before;
  take_eq = take_eq < 0 ? 0 : (take_eq > eq ? eq : take_eq);
  int o = block_exclusive_scan(gt + take_eq, scan_tmp) + gt_before + take_before;
  int e = 0;
  int32_t* dst = idx + (size_t)row * k;
  for (int i = s0; i < s1; ++i) {
    const uint32_t key = keys[i];
    bool take = key > T;
    if (key == T) { take = e < take_eq; ++e; }
    if (take) dst[o++] = lo + i;
  }
  cluster.sync();     // keep this CTA's shared memory alive until every peer has read it
}

bool topk_cluster_fits(int n) {
  const int slice = (n + kTopkClusterCtas - 1) / kTopkClusterCtas;
  return (size_t)slice * sizeof(uint32_t) <= 200 * 1024;
}

cudaError_t launch_topk_cluster(const float* scores, int rows, int n, int k, int32_t* idx,
                                cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int slice = (n + kTopkClusterCtas - 1) / kTopkClusterCtas;
  const size_t smem = (size_t)slice * sizeof(uint32_t);
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  dim3 grid(kTopkClusterCtas, rows);
  topk_cluster_kernel<<<grid, kTopkClusterThreads, smem, stream>>>(scores, n, k, idx);
  return cudaGetLastError();
}

}  // namespace sv
