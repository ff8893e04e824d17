// Query-aware retrieval scoring (decode phase).
//
// velog.io SparseVILA summary §3.2 "Query-Aware Token Selection": the current
// question's query rows are scored against every cached visual key; xllm-io
// review §三: Selected = TopK(Query . KV_Cache, k).  The score of visual token
// j for KV head g is sum_r sum_{h in g} q[r,h] . K[g,j]; by linearity the
// query rows and the group's heads are summed first (q_bar), so the kernel is
// one GEMV per (sequence, KV head) that streams the visual keys once.
//
// Memory-bound: each KV page of one head (16 tokens x d bf16, 2 or 4 KB,
// contiguous) is read by one warp with 16-byte loads; the per-lane partial dot
// products are folded with a butterfly reduce-scatter so the shuffle count per
// page is ~d/8 instead of 16 * log2(d/8).
#include "common.cuh"
#include "kernels.h"

namespace sv {

template <int D>
__global__ void __launch_bounds__(256)
retrieve_score_kernel(const uint16_t* __restrict__ q, int R, int H, int G,
                      const uint16_t* __restrict__ k_pool, int num_blocks, int Hkv,
                      const int32_t* __restrict__ block_table, int max_blocks, int n_vis,
                      int blocks_per_cta, float* __restrict__ scores, int* status) {
  constexpr int LPT = D / 8;        // lanes per token row (16 B each)
  constexpr int TPI = 32 / LPT;     // tokens per warp-wide load
  constexpr int NL = kBlockTokens / TPI;  // loads per lane per page
  static_assert(NL * 2 == LPT, "page fold assumes two lanes per reduced value");

  __shared__ float qbar[D];
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;

  // q_bar = sum over query rows r and the group's heads, fp32, fixed order.
  for (int e = tid; e < D; e += blockDim.x) {
    float acc = 0.f;
    for (int r = 0; r < R; ++r) {
      const uint16_t* row = q + (((size_t)b * R + r) * H + (size_t)g * G) * D + e;
      for (int hh = 0; hh < G; ++hh) acc += __uint_as_float((uint32_t)row[(size_t)hh * D] << 16);
    }
    qbar[e] = acc;
  }
  __syncthreads();

  float qv[8];
  const int dim0 = (lane % LPT) * 8;
#pragma unroll
  for (int e = 0; e < 8; ++e) qv[e] = qbar[dim0 + e];

  const int n_vblocks = (n_vis + kBlockTokens - 1) / kBlockTokens;
  const int blk_begin = blockIdx.x * blocks_per_cta;
  const int blk_end = min(n_vblocks, blk_begin + blocks_per_cta);
  const int32_t* bt = block_table + (size_t)b * max_blocks;
  float* out = scores + ((size_t)b * Hkv + g) * n_vis;
  // token held by this lane after the fold
  const int my_tok = ((lane % LPT) >> 1) * TPI + lane / LPT;

  for (int blk = blk_begin + warp; blk < blk_end; blk += nwarps) {
    const int page = __ldg(bt + blk);
    const bool ok = page >= 0 && page < num_blocks;
    if (!ok && lane == 0) flag_status(status, kStatusBadBlock);
    const uint16_t* base = k_pool + (((size_t)(ok ? page : 0) * Hkv + g) * kBlockTokens) * D;
    uint4 kv[NL];
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      if (ok) kv[i] = ld_stream16(base + (size_t)(lane + 32 * i) * 8);
      else kv[i] = make_uint4(0, 0, 0, 0);
    }
    float part[NL];
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const uint32_t w[4] = {kv[i].x, kv[i].y, kv[i].z, kv[i].w};
      float a = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        a = fmaf(qv[2 * c], bf16_lo(w[c]), a);
        a = fmaf(qv[2 * c + 1], bf16_hi(w[c]), a);
      }
      part[i] = a;
    }
    GroupReduce<NL, LPT>::run(part, lane);
    const int pos = blk * kBlockTokens + my_tok;
    if ((lane & 1) == 0 && pos < n_vis) out[pos] = part[0];
  }
}

cudaError_t launch_retrieve_score(const void* q, int R, int H, int G, const void* k_pool,
                                  int num_blocks, int Hkv, int D, const int32_t* block_table,
                                  int max_blocks, int n_vis, int batch, float* scores,
                                  int* status, int num_sms, cudaStream_t stream) {
  const int n_vblocks = (n_vis + kBlockTokens - 1) / kBlockTokens;
  const long long tasks = (long long)batch * Hkv * n_vblocks;
  // aim for ~16 resident warps' worth of pages per SM, at least 8 pages per CTA
  long long per = (tasks + (long long)num_sms * 16 - 1) / ((long long)num_sms * 16);
  int blocks_per_cta = (int)(per < 8 ? 8 : per);
  if (blocks_per_cta > n_vblocks) blocks_per_cta = n_vblocks;
  dim3 grid((n_vblocks + blocks_per_cta - 1) / blocks_per_cta, Hkv, batch);
  dim3 block(256);
  const uint16_t* qq = static_cast<const uint16_t*>(q);
  const uint16_t* kp = static_cast<const uint16_t*>(k_pool);
  if (D == 128)
    retrieve_score_kernel<128><<<grid, block, 0, stream>>>(qq, R, H, G, kp, num_blocks, Hkv,
        block_table, max_blocks, n_vis, blocks_per_cta, scores, status);
  else
    retrieve_score_kernel<64><<<grid, block, 0, stream>>>(qq, R, H, G, kp, num_blocks, Hkv,
        block_table, max_blocks, n_vis, blocks_per_cta, scores, status);
  return cudaGetLastError();
}

}  // namespace sv
