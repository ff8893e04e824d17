// Compaction of the kept prefill tokens (velog.io SparseVILA summary §2
// table: pruned prefill tokens are physically deleted; §3.2 on dense packing
// for coalesced reads).  out[b][t] = feat[b][idx[b][t]] for opaque rows of
// row_bytes (a multiple of 16): a pure HBM copy with 16-byte vectors, one
// warp per output row.
#include "common.cuh"
#include "kernels.h"

namespace sv {

__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ feat, int N, int k, int64_t row_vecs,
                   const int32_t* __restrict__ idx, uint4* __restrict__ out, long long rows,
                   int* status) {
  const int lane = threadIdx.x & 31;
  const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long r = warp; r < rows; r += nwarps) {
    const long long b = r / k;
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
                               const int32_t* idx, void* out, int* status, cudaStream_t stream) {
  const long long rows = (long long)B * k;
  if (rows == 0) return cudaSuccess;
  const int threads = 256;
  long long blocks = (rows + 7) / 8;
  if (blocks > 65535LL * 8) blocks = 65535LL * 8;
  gather_rows_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      static_cast<const uint4*>(feat), N, k, row_bytes / 16, idx, static_cast<uint4*>(out), rows,
      status);
  return cudaGetLastError();
}

}  // namespace sv
