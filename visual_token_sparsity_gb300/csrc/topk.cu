// Row-wise exact top-k with lowest-index tie-break and ascending output, as a
// stand-alone kernel (one CTA per row).
//
// The selection step of both SparseVILA phases (velog.io summary §3.1: prune
// the lowest-salience tokens; §3.2: keep the highest-scoring cached tokens
// active; xllm-io review §五 topk).  The algorithm lives in topk_block.cuh;
// rows of up to 52K scores are staged in shared memory, longer rows are
// re-read through L2 on every radix pass.
#include "common.cuh"
#include "kernels.h"
#include "topk_block.cuh"

namespace sv {

__global__ void __launch_bounds__(1024)
topk_rows_kernel(const float* __restrict__ scores, int n, int k, int32_t* __restrict__ idx,
                 int keys_in_smem, SeqLens lens, int rows_per_seq) {
  extern __shared__ __align__(16) uint32_t smem_keys[];
  __shared__ TopkShared ts;
  grid_dep_sync();
  const int row = blockIdx.x;
  int nr = n, kr = k;
  if (lens.any()) row_lengths(lens, row, rows_per_seq, n, k, nr, kr);
  int32_t* dst = idx + (size_t)row * k;
  if (kr > 0) block_topk_row(scores + (size_t)row * n, nr, kr, dst, keys_in_smem ? smem_keys : nullptr, ts);
  fill_unselected(dst, kr, k);
}

int topk_max_smem_keys() { return 52 * 1024; }   // 208 KB of keys

cudaError_t launch_topk_rows(const float* scores, int rows, int n, int k, int32_t* idx,
                             cudaStream_t stream, const SeqLens& lens, int rows_per_seq) {
  if (rows == 0) return cudaSuccess;
  const bool in_smem = n <= topk_max_smem_keys();
  const size_t smem = in_smem ? (size_t)n * sizeof(uint32_t) : 0;
  const int threads = n >= 16384 ? 1024 : (n >= 8192 ? 512 : 256);
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
  return launch_dependent(topk_rows_kernel, dim3(rows), dim3(threads), smem, stream, scores, n, k, idx,
                          in_smem ? 1 : 0, lens, rows_per_seq > 0 ? rows_per_seq : 1);
}

}  // namespace sv
