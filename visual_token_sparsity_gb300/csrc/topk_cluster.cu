// Row top-k for long rows on a thread-block cluster.
//
// The selection step of decode retrieval (velog.io SparseVILA summary §3.2)
// for long-video caches, where one (sequence, KV head) row holds tens of
// thousands of visual scores and a batch has only a few rows.  A cluster of
// kTopkClusterCtas CTAs owns one row; CTA r keeps the r-th slice of the row's
// order-preserving keys in its shared memory.  The cluster's smallest and
// largest keys fix the bits every key shares; each radix pass then builds a
// local 256-bin histogram of the next 8-bit window, and after a cluster
// barrier every CTA sums the cluster's histograms through distributed shared
// memory and picks the same digit (histograms are double-buffered, so one
// cluster barrier per pass is enough).  Passes stop once the selected bin
// holds exactly the keys still needed.  The output phase exchanges per-CTA
// (greater, equal) counts the same way, so the CTAs write disjoint ranges of
// the ascending index list, with ties broken towards the lower index exactly
// as in the single-CTA routine (topk_block.cuh).  The cluster barriers are
// hardware barriers over co-scheduled CTAs; nothing spins.
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
topk_cluster_kernel(const float* __restrict__ scores, int n_cap, int k_cap, int32_t* __restrict__ idx,
                    SeqLens lens, int rows_per_seq) {
  extern __shared__ uint32_t keys[];
  __shared__ int hist[2][256];    // double-buffered: peers read pass p's while pass p+1 fills the other
  __shared__ int total[256];
  __shared__ uint32_t scan_tmp[33];
  __shared__ uint32_t red_min[32], red_max[32];
  __shared__ uint32_t cta_min, cta_max;
  __shared__ int sel_digit, sel_above, sel_count;
  __shared__ int cnt[2];          // this CTA's (greater, equal) counts
  grid_dep_sync();
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int row = blockIdx.y;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  // this row's key count and selection size (the same for every CTA of the
  // cluster, so an empty selection leaves the cluster together)
  int n = n_cap, k = k_cap;
  if (lens.any()) row_lengths(lens, row, rows_per_seq, n_cap, k_cap, n, k);
  int32_t* dst = idx + (size_t)row * k_cap;
  if (rank == 0) fill_unselected(dst, k, k_cap);
  if (k <= 0) return;
  const int slice = (n + kTopkClusterCtas - 1) / kTopkClusterCtas;
  const int lo_i = min(n, rank * slice), hi_i = min(n, lo_i + slice);
  const int m = hi_i - lo_i;
  const float* src = scores + (size_t)row * n_cap + lo_i;

  // stage this CTA's keys (four independent loads in flight per thread) and
  // its smallest / largest key
  uint32_t lmin = 0xffffffffu, lmax = 0u;
  auto stage = [&](int i, float x) {
    const uint32_t key = order_key(x);
    keys[i] = key;
    lmin = min(lmin, key);
    lmax = max(lmax, key);
  };
  int i0 = tid;
  for (; i0 + 3 * nt < m; i0 += 4 * nt) {
    const float x0 = __ldcg(src + i0), x1 = __ldcg(src + i0 + nt);
    const float x2 = __ldcg(src + i0 + 2 * nt), x3 = __ldcg(src + i0 + 3 * nt);
    stage(i0, x0);
    stage(i0 + nt, x1);
    stage(i0 + 2 * nt, x2);
    stage(i0 + 3 * nt, x3);
  }
  for (; i0 < m; i0 += nt) stage(i0, __ldcg(src + i0));
  for (int i = tid; i < 512; i += nt) (&hist[0][0])[i] = 0;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    lmin = min(lmin, __shfl_xor_sync(0xffffffffu, lmin, o));
    lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, o));
  }
  if (lane == 0) {
    red_min[warp] = lmin;
    red_max[warp] = lmax;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = red_min[0], b = red_max[0];
    for (int w = 1; w < nw; ++w) {
      a = min(a, red_min[w]);
      b = max(b, red_max[w]);
    }
    cta_min = a;   // an empty slice contributes (max, 0): neutral
    cta_max = b;
  }
  cluster.sync();
  uint32_t kmin = 0xffffffffu, kmax = 0u;
#pragma unroll
  for (int r = 0; r < kTopkClusterCtas; ++r) {
    kmin = min(kmin, *cluster.map_shared_rank(&cta_min, r));
    kmax = max(kmax, *cluster.map_shared_rank(&cta_max, r));
  }

  uint32_t prefix, pmask;
  int remaining = k;
  const uint32_t diff = kmin ^ kmax;
  if (diff == 0) {
    prefix = kmin;
    pmask = 0xffffffffu;
  } else {
    const int top = 31 - __clz(diff);
    pmask = top == 31 ? 0u : ~((2u << top) - 1u);
    prefix = kmin & pmask;
    int hi = top + 1;
#pragma unroll 1
    for (int pass = 0; hi > 0; ++pass) {
      const int lo = hi > 8 ? hi - 8 : 0;
      const uint32_t wmask = (1u << (hi - lo)) - 1u;
      int* hcur = hist[pass & 1];
      for (int i = tid; i < m; i += nt) {
        const uint32_t key = keys[i];
        if ((key & pmask) == prefix) atomicAdd(&hcur[(key >> lo) & wmask], 1);
      }
      cluster.sync();                                   // all local histograms complete
      for (int b = tid; b < 256; b += nt) {
        int s = 0;
#pragma unroll
        for (int r = 0; r < kTopkClusterCtas; ++r) s += cluster.map_shared_rank(hcur, r)[b];
        total[b] = s;
      }
      // the other buffer was last read by peers before this pass's barrier
      for (int i = tid; i < 256; i += nt) hist[(pass + 1) & 1][i] = 0;
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
            if (run + c[j] >= remaining) {
              sel_digit = 255 - 8 * tid - j;
              sel_above = run;
              sel_count = c[j];
              break;
            }
            run += c[j];
          }
        }
      }
      __syncthreads();
      prefix |= (uint32_t)sel_digit << lo;
      pmask |= wmask << lo;
      remaining -= sel_above;
      const int cnt_sel = sel_count;
      __syncthreads();          // total / sel_* are rewritten by the next pass
      if (cnt_sel == remaining || lo == 0) break;
      hi = lo;
    }
  }

  // this CTA's counts, then the counts of the CTAs before it in the row
  const int seg = (m + nt - 1) / nt;
  const int s0 = min(m, tid * seg), s1 = min(m, s0 + seg);
  int gt = 0, eq = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t kp = keys[i] & pmask;
    gt += kp > prefix;
    eq += kp == prefix;
  }
  if (tid == 0) cnt[0] = cnt[1] = 0;
  __syncthreads();
  int w_gt = gt, w_eq = eq;
#pragma unroll
  for (int o2 = 16; o2 >= 1; o2 >>= 1) {
    w_gt += __shfl_xor_sync(0xffffffffu, w_gt, o2);
    w_eq += __shfl_xor_sync(0xffffffffu, w_eq, o2);
  }
  if (lane == 0) { atomicAdd(&cnt[0], w_gt); atomicAdd(&cnt[1], w_eq); }
  cluster.sync();
  int gt_before = 0, eq_before_cta = 0;
  for (int r = 0; r < rank; ++r) {
    const int* rc = cluster.map_shared_rank(cnt, r);
    gt_before += rc[0];
    eq_before_cta += rc[1];
  }
  // within the CTA: one scan of the packed (greater, equal) pair (a slice
  // holds fewer than 65536 keys)
  const uint32_t packed = block_exclusive_scan<uint32_t>(((uint32_t)gt << 16) | (uint32_t)eq, scan_tmp);
  const int eq_before = (int)(packed & 0xffffu) + eq_before_cta;
  int take_eq = remaining - eq_before;
  take_eq = take_eq < 0 ? 0 : (take_eq > eq ? eq : take_eq);
  int o = gt_before + (int)(packed >> 16) + min(eq_before, remaining);
  int e = 0;
  for (int i = s0; i < s1; ++i) {
    const uint32_t kp = keys[i] & pmask;
    bool take = kp > prefix;
    if (kp == prefix) {
      take = e < take_eq;
      ++e;
    }
    if (take) dst[o++] = lo_i + i;
  }
  cluster.sync();     // keep this CTA's shared memory alive until every peer has read it
}

bool topk_cluster_fits(int n) {
  const int slice = (n + kTopkClusterCtas - 1) / kTopkClusterCtas;
  return (size_t)slice * sizeof(uint32_t) <= 200 * 1024;
}

// Short rows keep one CTA per row: below ~16K keys a cluster's barriers and
// DSMEM exchanges cost more than the 8x wider slice saves.
bool topk_prefers_cluster(int n) { return n > 16384 && topk_cluster_fits(n); }

cudaError_t launch_topk_cluster(const float* scores, int rows, int n, int k, int32_t* idx,
                                cudaStream_t stream, const SeqLens& lens, int rows_per_seq) {
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
  return launch_dependent(topk_cluster_kernel, grid, dim3(kTopkClusterThreads), smem, stream, scores, n, k, idx,
                          lens, rows_per_seq > 0 ? rows_per_seq : 1);
}

}  // namespace sv
