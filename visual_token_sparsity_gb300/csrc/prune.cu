// Compaction of the kept prefill tokens (velog.io SparseVILA summary §2
// table: pruned prefill tokens are physically deleted; §3.2 on dense packing
// for coalesced reads).  out[b][t] = feat[b][idx[b][t]] for opaque rows of
// row_bytes (a multiple of 16): a pure HBM copy with 16-byte vectors.
#include "common.cuh"
#include "kernels.h"
#include "topk_block.cuh"

namespace sv {

// The output is one flat array of 16-byte vectors (rows x row_vecs); each
// warp copies a contiguous stretch of kGatherU x 32 of them, so a lane issues
// kGatherU independent loads before its first store whatever the row size,
// and consecutive lanes touch consecutive bytes of the same source row.
// counts (optional): frame b has counts[b] valid rows; later slots are skipped
constexpr int kGatherU = 8;
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ feat, int N, int k, int row_vecs,
                   const int32_t* __restrict__ idx, uint4* __restrict__ out, long long total,
                   const int32_t* __restrict__ counts, int* status) {
  grid_dep_sync();
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long base = warp * (32 * kGatherU); base < total; base += nwarps * (32 * kGatherU)) {
    // this lane's first vector: row r (slot rs of frame b), column c; the
    // later ones follow 32 vectors apart
    const long long i0 = base + lane;
    long long r = i0 / row_vecs;
    int c = (int)(i0 - r * row_vecs);
    long long b = r / k;
    int rs = (int)(r - b * k);
    uint4 v[kGatherU];
    long long dst[kGatherU];
#pragma unroll
    for (int u = 0; u < kGatherU; ++u) {
      const long long i = i0 + u * 32;
      dst[u] = -1;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (i < total && !(counts && rs >= __ldg(counts + b))) {
        dst[u] = i;
        const int src = __ldg(idx + r);
        if (src < 0 || src >= N) {
          if (c == 0) flag_status(status, kStatusBadIndex);   // the slot is written with zeros
        } else {
          v[u] = ld_stream16(feat + (b * N + src) * row_vecs + c);
        }
      }
      c += 32;
      while (c >= row_vecs) {
        c -= row_vecs;
        ++r;
        if (++rs == k) {
          rs = 0;
          ++b;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kGatherU; ++u)
      if (dst[u] >= 0) out[dst[u]] = v[u];
  }
}

cudaError_t launch_gather_rows(const void* feat, int B, int N, int k, int64_t row_bytes,
                               const int32_t* idx, void* out, int* status, cudaStream_t stream,
                               const int32_t* counts) {
  const long long rows = (long long)B * k;
  const long long row_vecs = row_bytes / 16;
  if (rows == 0 || row_vecs == 0) return cudaSuccess;
  if (row_vecs > 0x7fffffffLL) return cudaErrorInvalidValue;
  const long long total = rows * row_vecs;
  const int threads = 256;
  const long long per_block = (long long)threads * kGatherU;
  long long blocks = (total + per_block - 1) / per_block;
  if (blocks > 65535LL * 16) blocks = 65535LL * 16;
  return launch_dependent(gather_rows_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream,
                          static_cast<const uint4*>(feat), N, k, (int)row_vecs, idx, static_cast<uint4*>(out), total,
                          counts, status);
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
  grid_dep_sync();
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
  return launch_dependent(threshold_select_kernel, dim3(B), dim3(512), 0, stream, sal, N, threshold, idx, count);
}

}  // namespace sv
