// Query-agnostic salience for encoders with summary tokens.
//
// velog.io SparseVILA summary §3.1 (encoder-type table): with one summary
// token (CLIP) a token's importance is the attention it contributes to the
// global embedding, i.e. the summary token's attention row; with several
// (RADIO) it is the mean attention toward them.  With the R summary tokens
// leading the sequence, per frame b:
//   s[b][j] = 1/(H R) sum_h sum_{r<R} exp(scale q_r.k_j - lse_r),
//   lse_r   = log sum_j exp(scale q_r.k_j)   (over all N tokens).
//
// Only R rows of the attention map are needed, so the work is a few GEMVs
// per head and HBM-bound on K: one CTA per (frame, head) reads K once with
// 16-byte loads (d/8 lanes per token), keeps the R x N logits (log2 domain)
// in shared memory, takes each row's log-sum-exp with one warp per row, and
// writes per-key column sums; a second kernel averages the heads in order.
#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {
// 128 threads: more independent CTAs per SM overlap one CTA's load phase with
// another's row reductions (measured faster than 64, 256 or 512; staging the
// head's K through bulk copies into shared memory, or splitting a head over
// several CTAs, was slower)
constexpr int kSumThreads = 128;
constexpr int kSumWarps = kSumThreads / 32;

size_t summary_smem(int N, int d, int R) { return ((size_t)R * d + (size_t)R * N + 2 * (size_t)R) * sizeof(float); }
}  // namespace

// One summary row (CLIP): the query row stays in registers across the key
// loop, six token groups per lane are in flight and the kernel is
// register-capped for eight CTAs per SM; several rows (RADIO): four groups,
// uncapped (measured on the 256-frame CLIP shape: one row, 6 groups, 8 CTAs
// 59.0 us; 4 groups 60.7 us; 8 groups at 80 registers 69.7 us; the generic
// loop over R rows 70.5 us)
template <bool kOneRow>
__global__ void __launch_bounds__(kSumThreads, kOneRow ? 8 : 1)
summary_colsum_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ k, int N, int d, int R,
                      float sl2, float* __restrict__ colsum) {
  extern __shared__ float sm[];
  grid_dep_sync();
  float* qs = sm;                       // [R][d], scaled by scale * log2(e)
  float* z = qs + (size_t)R * d;        // [R][N] logits, log2 domain
  float* lse = z + (size_t)R * N;       // [R]
  const size_t unit = blockIdx.x;
  const uint16_t* qb = q + unit * (size_t)N * d;
  const uint16_t* kb = k + unit * (size_t)N * d;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  for (int i = tid; i < R * d; i += kSumThreads) qs[i] = __uint_as_float((uint32_t)qb[i] << 16) * sl2;
  __syncthreads();

  // logits: a group of lpt lanes (cpr = d / 8 rounded up to a power of two)
  // holds one key row, 16 bytes per lane; lanes past the row contribute 0
  const int cpr = d >> 3;                          // d <= 256: cpr <= 32
  int lpt = 1;
  while (lpt < cpr) lpt <<= 1;
  const int tpw = 32 / lpt;                        // tokens per warp step
  const int sub = lane % lpt, slot = lane / lpt;
  // kSumU token groups per iteration, all loads in flight before the first
  // dot product needs one; the raw 16-byte words stay packed (4 registers per
  // group) until they are used
  constexpr int kU = kOneRow ? 6 : 4;
  const int stride = kSumWarps * tpw;
  for (int j0 = warp * tpw; j0 < N; j0 += kU * stride) {
    uint4 raw[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int j = j0 + u * stride + slot;
      raw[u] = (j < N && sub < cpr) ? ld_stream16(kb + (size_t)j * d + sub * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
    const int nr = kOneRow ? 1 : R;
    for (int r = 0; r < nr; ++r) {
      float qv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (sub < cpr) {
        const float* qr = qs + (size_t)r * d + sub * 8;
#pragma unroll
        for (int e = 0; e < 8; ++e) qv[e] = qr[e];
      }
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
        float acc = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          acc = fmaf(qv[2 * c], bf16_lo(w[c]), acc);
          acc = fmaf(qv[2 * c + 1], bf16_hi(w[c]), acc);
        }
        for (int o = lpt >> 1; o >= 1; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        const int j = j0 + u * stride + slot;
        if (j < N && sub == 0) z[(size_t)r * N + j] = acc;
      }
    }
  }
  __syncthreads();

  // per summary row: log-sum-exp over all N keys (log2 domain), one warp per row
  for (int r = warp; r < R; r += kSumWarps) {
    const float* zr = z + (size_t)r * N;
    float m = -INFINITY;
    for (int j = lane; j < N; j += 32) m = fmaxf(m, zr[j]);
    m = warp_max(m);
    float l = 0.f;
    for (int j = lane; j < N; j += 32) l += fast_exp2(zr[j] - m);
    l = warp_sum(l);
    if (lane == 0) lse[r] = m + __log2f(l);
  }
  __syncthreads();

  float* out = colsum + unit * (size_t)N;
  for (int j = tid; j < N; j += kSumThreads) {
    float c = 0.f;
    for (int r = 0; r < R; ++r) c += fast_exp2(z[(size_t)r * N + j] - lse[r]);
    out[j] = c;
  }
}

size_t summary_smem_bytes(int N, int d, int R) { return summary_smem(N, d, R); }

cudaError_t launch_summary_salience(const void* q, const void* k, int B, int H, int N, int d, int R,
                                    float scale, float* salience, float* colsum, cudaStream_t stream) {
  const long long units = (long long)B * H;
  if (units == 0) return cudaSuccess;
  const size_t smem = summary_smem(N, d, R);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(summary_colsum_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(summary_colsum_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  auto kern = R == 1 ? summary_colsum_kernel<true> : summary_colsum_kernel<false>;
  cudaError_t e = launch_dependent(kern, dim3((unsigned)units), dim3(kSumThreads), smem, stream,
                                   static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k), N, d, R,
                                   scale * kLog2e, colsum);
  if (e != cudaSuccess) return e;
  return launch_head_mean(colsum, B, H, N, 1.0f / ((float)H * (float)R), salience, stream);
}

}  // namespace sv
