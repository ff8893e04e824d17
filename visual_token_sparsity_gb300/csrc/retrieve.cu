// Query-aware retrieval (decode phase): scoring GEMV fused with the top-k.
//
// velog.io SparseVILA summary §3.2 "Query-Aware Token Selection": the current
// question's query rows are scored against every cached visual key; xllm-io
// review §三: Selected = TopK(Query . KV_Cache, k).  The score of visual token
// j for KV head g is sum_r sum_{h in g} q[r,h] . K[g,j]; by linearity the
// query rows and the group's heads are summed first (q_bar), so scoring is one
// GEMV per (sequence, KV head) row that streams the visual keys once.
//
// Memory-bound.  A CTA scores a contiguous run of KV pages of one row; each
// warp reads whole pages (16 tokens x d bf16, 2 or 4 KB, contiguous) with
// 16-byte loads and folds the per-lane partial dot products with a butterfly
// reduce-scatter (~d/8 shuffles per page).  One page in flight per warp
// measured faster than a register-prefetched second page at 104 registers;
// capping the kernel at 48 registers (5 CTAs, 40 warps per SM; the fused
// top-k spills a few words) measured 12 % faster than 64 registers (4 CTAs)
// on LLaVA-NeXT rows and slower at 6 or 8 CTAs.  For calls with a few rows
// the CTA that finishes a row last (a device-scope counter per row, no
// waiting) runs the exact block top-k on that row's scores while other rows
// are still streaming, so no separate selection kernel is launched; calls
// with many rows, or rows too long for shared memory, select in a separate
// top-k kernel.
#include "common.cuh"
#include "kernels.h"
#include "topk_block.cuh"

namespace sv {

#ifndef SV_RET_PREFETCH
#define SV_RET_PREFETCH 0      // 1: keep the next page in flight (more registers, fewer warps)
#endif
#ifndef SV_RET_THREADS
#define SV_RET_THREADS 256
#endif
#ifndef SV_RET_WAVES
#define SV_RET_WAVES 20        // target CTAs = SMs x this (12 / 16 / 20 / 24 / 32 measured: 20 best)
#endif
#ifndef SV_RET_MINB
#define SV_RET_MINB 5          // register cap: 5 resident CTAs (40 warps) per SM
#endif

namespace {
constexpr int kRetrieveThreads = SV_RET_THREADS;
constexpr int kFuseMaxN = 11264;   // keys in dynamic shared memory (44 KB; static + dynamic < 48 KB)
// The fused selection pays off for a few rows, where it overlaps the
// streaming of the others; with many rows the last wave's selections form a
// tail, and a separate top-k launch (overlapped with the scoring kernel's
// drain) measured faster: LLaVA-NeXT rows, 128 and 512 rows 2.3-2.7 us per
// call faster separate, 32 rows 1.4 us faster fused.
constexpr int kFuseMaxRows = 64;
}  // namespace

template <int D>
__global__ void __launch_bounds__(kRetrieveThreads, SV_RET_MINB)
retrieve_score_kernel(const uint16_t* __restrict__ q, int R, int H, int G,
                      const uint16_t* __restrict__ k_pool, int num_blocks, int Hkv,
                      const int32_t* __restrict__ block_table, int max_blocks, int n_vis,
                      int blocks_per_cta, float* __restrict__ scores, int* status,
                      int* row_done, int k, int32_t* __restrict__ vis_idx, SeqLens lens, int n_text) {
  constexpr int LPT = D / 8;        // lanes per token row (16 B each)
  constexpr int TPI = 32 / LPT;     // tokens per warp-wide load
  constexpr int NL = kBlockTokens / TPI;  // loads per lane per page
  static_assert(NL * 2 == LPT, "page fold assumes two lanes per reduced value");

  extern __shared__ __align__(16) uint32_t topk_keys[];
  __shared__ float qbar[D];
  __shared__ TopkShared ts;
  __shared__ int s_last;
  grid_dep_sync();
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int row = b * Hkv + g;
  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;

  // this sequence's visual count and selection size (n_vis and k are the
  // capacities: the strides of scores and vis_idx)
  int nv = n_vis, nt, kb = k;
  if (lens.any() && !seq_lengths(lens, b, n_vis, n_text, k, nv, nt, kb) && tid == 0 && blockIdx.x == 0)
    flag_status(status, kStatusBadLength);
  const int n_vblocks = (nv + kBlockTokens - 1) / kBlockTokens;
  const int blk_begin = blockIdx.x * blocks_per_cta;
  const int blk_end = min(n_vblocks, blk_begin + blocks_per_cta);
  const int32_t* bt = block_table + (size_t)b * max_blocks;
  float* out = scores + (size_t)row * n_vis;
  // token held by this lane after the fold
  const int my_tok = ((lane % LPT) >> 1) * TPI + lane / LPT;

  auto load_page = [&](int blk, uint4* kv) {
    const int page = __ldg(bt + blk);
    const bool ok = page >= 0 && page < num_blocks;
    if (!ok && lane == 0) flag_status(status, kStatusBadBlock);
    const uint16_t* base = k_pool + (((size_t)(ok ? page : 0) * Hkv + g) * kBlockTokens) * D;
#pragma unroll
    for (int i = 0; i < NL; ++i)
      kv[i] = ok ? ld_stream16(base + (size_t)(lane + 32 * i) * 8) : make_uint4(0, 0, 0, 0);
  };

  // the first page's loads are issued before the q_bar prologue so that its
  // latency overlaps the prologue's loads and barrier
  uint4 cur[NL], nxt[NL];
  const int blk0 = blk_begin + warp;
  if (blk0 < blk_end) load_page(blk0, cur);

  // q_bar = sum over query rows r and the group's heads, fp32, fixed order.
  for (int e = tid; e < D; e += blockDim.x) {
    float acc = 0.f;
    for (int r = 0; r < R; ++r) {
      const uint16_t* qr = q + (((size_t)b * R + r) * H + (size_t)g * G) * D + e;
      for (int hh = 0; hh < G; ++hh) acc += __uint_as_float((uint32_t)qr[(size_t)hh * D] << 16);
    }
    qbar[e] = acc;
  }
  __syncthreads();

  float qv[8];
  const int dim0 = (lane % LPT) * 8;
#pragma unroll
  for (int e = 0; e < 8; ++e) qv[e] = qbar[dim0 + e];

  int blk = blk0;
  for (; blk < blk_end; blk += nwarps) {
    if (!SV_RET_PREFETCH && blk != blk0) load_page(blk, cur);
    else if (SV_RET_PREFETCH && blk + nwarps < blk_end) load_page(blk + nwarps, nxt);
    float part[NL];
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const uint32_t w[4] = {cur[i].x, cur[i].y, cur[i].z, cur[i].w};
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
    if ((lane & 1) == 0 && pos < nv) out[pos] = part[0];
    if (SV_RET_PREFETCH) {
#pragma unroll
      for (int i = 0; i < NL; ++i) cur[i] = nxt[i];
    }
  }

  if (row_done == nullptr) return;
  // last CTA of this row selects its top-k
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(row_done + row, 1) == (int)gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  int32_t* dst = vis_idx + (size_t)row * k;
  if (kb > 0) block_topk_row(out, nv, kb, dst, topk_keys, ts);
  fill_unselected(dst, kb, k);
  if (tid == 0) row_done[row] = 0;   // ready for the next call
}

bool retrieve_fuses_topk(int rows, int n_vis) { return rows <= kFuseMaxRows && n_vis <= kFuseMaxN; }

cudaError_t launch_retrieve(const void* q, int R, int H, int G, const void* k_pool, int num_blocks,
                            int Hkv, int D, const int32_t* block_table, int max_blocks, int n_vis,
                            int batch, float* scores, int* status, int num_sms, int* row_done, int k,
                            int32_t* vis_idx, cudaStream_t stream, const SeqLens& lens, int n_text) {
  const int n_vblocks = (n_vis + kBlockTokens - 1) / kBlockTokens;
  const int rows = batch * Hkv;
  // about two waves of 8-warp CTAs over the GPU, at least one page per warp
  const long long target = (long long)num_sms * SV_RET_WAVES;
  long long chunks = (target + rows - 1) / rows;
  int per = (int)((n_vblocks + chunks - 1) / chunks);
  // whole pages per warp (a multiple of the CTA's warps), so that every warp
  // of a CTA streams the same number of pages: rounded down, at least one
  // page per warp (measured against the unrounded split: LLaVA-NeXT B16 step
  // 4.572 -> 4.533 ms, B4 1.709 -> 1.662 ms, LongVILA B8 3.722 -> 3.710 ms)
  constexpr int kW = kRetrieveThreads / 32;
  per = per / kW * kW;
  if (per < kW) per = kW;
  if (per > n_vblocks) per = n_vblocks;
  const int grid_x = (n_vblocks + per - 1) / per;
  const bool fuse = row_done != nullptr && retrieve_fuses_topk(rows, n_vis);
  const size_t smem = fuse ? (size_t)n_vis * sizeof(uint32_t) : 0;
  dim3 grid(grid_x, Hkv, batch);
  const uint16_t* qq = static_cast<const uint16_t*>(q);
  const uint16_t* kp = static_cast<const uint16_t*>(k_pool);
  int* done = fuse ? row_done : nullptr;
  cudaError_t e =
      D == 128 ? launch_dependent(retrieve_score_kernel<128>, grid, dim3(kRetrieveThreads), smem, stream, qq, R, H, G,
                                  kp, num_blocks, Hkv, block_table, max_blocks, n_vis, per, scores, status, done, k,
                                  vis_idx, lens, n_text)
               : launch_dependent(retrieve_score_kernel<64>, grid, dim3(kRetrieveThreads), smem, stream, qq, R, H, G,
                                  kp, num_blocks, Hkv, block_table, max_blocks, n_vis, per, scores, status, done, k,
                                  vis_idx, lens, n_text);
  if (e != cudaSuccess || fuse) return e;
  if (topk_prefers_cluster(n_vis))
    return launch_topk_cluster(scores, rows, n_vis, k, vis_idx, stream, lens, Hkv);
  return launch_topk_rows(scores, rows, n_vis, k, vis_idx, stream, lens, Hkv);
}

}  // namespace sv
