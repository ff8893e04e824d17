// Compaction of the kept prefill tokens (velog.io SparseVILA summary §2
// table: pruned prefill tokens are physically deleted; §3.2 on dense packing
// for coalesced reads).  out[b][t] = feat[b][idx[b][t]] for opaque rows of
// row_bytes (a multiple of 16): a pure HBM copy with 16-byte vectors, one
// warp per output row.
#include "common.cuh"
#include "kernels.h"
#include "topk_block.cuh"

namespace sv {

// counts (optional): frame b has counts[b] valid rows; later slots are skipped
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ feat, int N, int k, int64_t row_vecs,
                   const int32_t* __restrict__ idx, uint4* __restrict__ out, long long rows,
                   const int32_t* __restrict__ counts, int* status) {
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r = warp; r < rows; r += nwarps) {
    const long long b = r / k;
    if (counts && r - b * k >= __ldg(counts + b)) continue;
    const int src = __ldg(idx + r);
    uint4* dst = out + r * row_vecs;
    if (src < 0 || src >= N) {
      if (lane == 0) flag_status(status, kStatusBadIndex);
      for (int64_t v = lane; v < row_vecs; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
      continue;
    }
    const uint4* s = feat + (b * N + src) * row_vecs;
    int64_t v = lane;
    for (; v + 96 < row_vecs; v += 128) {
      const uint4 a0 = ld_stream16(s + v), a1 = ld_stream16(s + v + 32);
      const uint4 a2 = ld_stream16(s + v + 64), a3 = ld_stream16(s + v + 96);
      dst[v] = a0; dst[v + 32] = a1; dst[v + 64] = a2; dst[v + 96] = a3;
    }
    for (; v < row_vecs; v += 32) dst[v] = ld_stream16(s + v);
  }
}

cudaError_t launch_gather_rows(const void* feat, int B, int N, int k, int64_t row_bytes,
                               const int32_t* idx, void* out, int* status, cudaStream_t stream,
                               const int32_t* counts) {
  const long long rows = (long long)B * k;
  if (rows == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (rows + 7) / 8;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  gather_rows_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      static_cast<const uint4*>(feat), N, k, row_bytes / 16, idx, static_cast<uint4*>(out), rows,
      counts, status);
  return cudaGetLastError();
}

// Threshold prune (xllm-io review §五 query_agnostic_pruning: keep the tokens
// whose salience exceeds the threshold, in order).  One CTA per frame:
// contiguous per-thread segments, a block scan of the kept counts, then the
// kept indices in ascending order; slots past the count get -1.
__global__ void __launch_bounds__(512)
threshold_select_kernel(const float* __restrict__ sal, int N, float threshold, int32_t* __restrict__ idx,
                        int32_t* __restrict__ count) {
  __shared__ int scan_tmp[33];
  __shared__ int s_total;
  const int b = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
  const float* s = sal + (size_t)b * N;
  int32_t* dst = idx + (size_t)b * N;
  const int seg = (N + nt - 1) / nt;
  const int s0 = min(N, tid * seg), s1 = min(N, s0 + seg);
  int kept = 0;
  for (int i = s0; i < s1; ++i) kept += __ldg(s + i) > threshold;
  int o = block_exclusive_scan<int>(kept, scan_tmp);
  if (tid == nt - 1) {
    s_total = o + kept;
    count[b] = o + kept;
  }
  for (int i = s0; i < s1; ++i)
    if (__ldg(s + i) > threshold) dst[o++] = i;
  __syncthreads();
  for (int i = s_total + tid; i < N; i += nt) dst[i] = -1;
}

cudaError_t launch_threshold_select(const float* sal, int B, int N, float threshold, int32_t* idx, int32_t* count,
                                    cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  threshold_select_kernel<<<B, 512, 0, stream>>>(sal, N, threshold, idx, count);
  return cudaGetLastError();
}

}  // namespace sv
