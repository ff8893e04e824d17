// Sparse decode attention for grouped-query heads (G >= 3) on warp-level
// tensor-core MMAs.
//
// Same computation as attn.cu (velog.io SparseVILA summary §3.2 and §4.5
// kernel table: attention of the decode query over the retrieved visual
// tokens plus all text tokens, read from the paged cache): for the G query
// heads of one KV head the score and value products are small matrix
// products, S = Q K^T (G x 16 tokens) and O += P V, so the G heads share every
// K/V tile through mma.sync (heads padded to the 16 rows of an m16n8k16 tile)
// instead of G separate dot products per token.  The kernel stays bound by
// HBM: each warp streams its split's gathered token rows through a 3-stage
// cp.async ring in (XOR-swizzled) shared memory, reads MMA fragments with
// ldmatrix, keeps the softmax state in fp32 (log2 domain) and converts P to
// bf16 only as the A operand of the PV product.
#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {

#ifndef SV_MMA_WARPS
#define SV_MMA_WARPS 2
#endif
#ifndef SV_MMA_STAGES
#define SV_MMA_STAGES 3
#endif
// Three stages (two sub-tiles in flight while one is processed): 48 KB of
// shared memory per 2-warp CTA, four CTAs (eight warps) per SM.  Measured
// against two stages with 4-warp CTAs (twelve warps per SM) and against
// 1-, 3- and 4-stage, 1- to 3-warp shapes: 2-5 % faster on every GQA shape
// tried (LongVILA-7B batch 8 / 1, the same model at 16 frames).
constexpr int kMmaWarps = SV_MMA_WARPS;
constexpr int kMmaStages = SV_MMA_STAGES;
constexpr int kSubTile = 16;      // tokens per MMA step
constexpr uint32_t kNoRowM = kNoRowId;


__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
// D = A (16x16 bf16, row) * B (16x8 bf16, col) + D, fp32
__device__ __forceinline__ void mma_bf16_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return f32_to_bf16_bits(lo) | (f32_to_bf16_bits(hi) << 16);
}

}  // namespace

// One warp per (sequence, KV head, token split); each warp owns a private
// kMmaStages-deep ring of K and V sub-tiles in shared memory.
// APPEND: the fused append-and-attend variant (k_new / v_new set), a separate
// instantiation.
template <int D, bool APPEND>
__global__ void __launch_bounds__(kMmaWarps * 32)
sparse_attn_mma_kernel(const uint16_t* __restrict__ q, int H, int G,
                       const uint16_t* __restrict__ k_pool, const uint16_t* __restrict__ v_pool,
                       int num_blocks, int Hkv, const int32_t* __restrict__ block_table,
                       int max_blocks, const int32_t* __restrict__ vis_idx, int k_vis, int n_vis,
                       int n_text, float scale_log2, int batch, int nsplit, int chunk,
                       float* __restrict__ part_ml, float* __restrict__ part_o, int* status,
                       int* split_done, uint16_t* __restrict__ out, float* __restrict__ lse,
                       SeqLens lens, const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                       uint16_t* k_store, uint16_t* v_store) {
  constexpr int CPR = D / 8;                         // 16-byte chunks per token row
  constexpr int KSTEPS = D / 16;
  constexpr int NT_O = D / 8;                        // output n-tiles (8 dims each)
  constexpr int TILE_BYTES = kSubTile * D * 2;       // one K or V sub-tile
  extern __shared__ __align__(128) uint8_t smem[];
  grid_dep_sync();
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  uint8_t* my = smem + (size_t)wid * kMmaStages * 2 * TILE_BYTES;

  const long long w = (long long)blockIdx.x * kMmaWarps + wid;
  if (w >= (long long)batch * Hkv * nsplit) return;
  const int split = (int)(w % nsplit);
  const int bg = (int)(w / nsplit);
  const int b = bg / Hkv, g = bg % Hkv;
  // this sequence's counts (capacities with per-sequence lengths)
  int nv, nt, kb;
  const bool seq_ok = attn_lengths(lens, vis_idx != nullptr, b, n_vis, n_text, k_vis,
                                   lane == 0 && split == 0 && g == 0, status, nv, nt, kb);
  // a fused append adds the new token (cache position nv + nt) as the last one
  const bool append = APPEND && seq_ok;
  const int T = kb + nt + (append ? 1 : 0);
  const int t_begin = split * chunk;
  const int t_end = min(T, t_begin + chunk);
  const int32_t* bt = block_table + (size_t)b * max_blocks;
  if (append && split == 0)
    store_new_token(k_store, v_store, k_new, v_new, bt, num_blocks, Hkv, D, b, g, nv + nt, lane);
  const int32_t* vrow = vis_idx ? vis_idx + (size_t)bg * k_vis : nullptr;

  // Q fragments (A operand, rows = heads of the group, zero beyond G)
  uint32_t qa[KSTEPS][4];
  {
    const int r0 = lane >> 2, c0 = (lane & 3) * 2;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
      for (int hlf = 0; hlf < 2; ++hlf) {          // rows r0 and r0 + 8
        const int hrow = r0 + 8 * hlf;
        uint32_t lo = 0, hi = 0;
        if (hrow < G) {
          const uint16_t* qp = q + ((size_t)b * H + (size_t)g * G + hrow) * D + ks * 16 + c0;
          lo = *reinterpret_cast<const uint32_t*>(qp);
          hi = *reinterpret_cast<const uint32_t*>(qp + 8);
        }
        qa[ks][hlf] = lo;        // a0 / a1: cols c0, c0+1
        qa[ks][2 + hlf] = hi;    // a2 / a3: cols c0+8, c0+9
      }
    }
  }

  // issue the cp.async copies of one sub-tile into stage s; returns the row ids
  auto issue = [&](int t0, int s, uint32_t rowid) -> uint32_t {
    (void)t0;
    const uint32_t kbase = smem_u32(my + (size_t)s * 2 * TILE_BYTES);
    const uint32_t vbase = kbase + TILE_BYTES;
#pragma unroll
    for (int i = 0; i < kSubTile * CPR / 32; ++i) {
      const int j = lane + 32 * i;
      const int tok = j / CPR, c = j % CPR;
      const uint32_t r = __shfl_sync(0xffffffffu, rowid, tok);
      const bool ok = r != kNoRowM;
      const bool fresh = APPEND && r == kNewRowId;   // the appended token: from k_new / v_new
      const size_t off = fresh ? (size_t)bg * D + c * 8 : (ok ? (size_t)r * D + c * 8 : 0);
      const uint32_t dst = (uint32_t)(tok * D * 2 + ((c ^ (tok & 7)) * 16));
      cp_async16(kbase + dst, (fresh ? k_new : k_pool) + off, ok ? 16u : 0u);
      cp_async16(vbase + dst, (fresh ? v_new : v_pool) + off, ok ? 16u : 0u);
    }
    cp_async_commit();
    return rowid;
  };

  float m_r[2] = {-INFINITY, -INFINITY};   // rows lane/4 and lane/4 + 8
  float l_r[2] = {0.f, 0.f};
  float o[NT_O][4];
#pragma unroll
  for (int j = 0; j < NT_O; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

  const int nsub = (t_end - t_begin + kSubTile - 1) / kSubTile;
  uint32_t rows[kMmaStages];
  // Row ids of 128-token blocks (8 sub-tiles) come through a software
  // pipeline: a block's visual indices are loaded two blocks ahead, its
  // page-table entries one block ahead, and its row ids are formed when its
  // first sub-tile is issued, so neither dependent round trip stalls the
  // stream (only the first block's two wait, before the first copy).
  int pos_a[4], pg_a[4];                  // block j + 1: checked positions, pages in flight
  int pos_b[4];                           // block j + 2: raw visual indices in flight
  uint32_t blk_cur[4];                    // block j: row ids
#pragma unroll
  for (int q4 = 0; q4 < 4; ++q4) { pos_a[q4] = pg_a[q4] = pos_b[q4] = -1; blk_cur[q4] = kNoRowM; }
  auto load_idx = [&](int t0, int* p) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int tok = t0 + 32 * q4 + lane;
      p[q4] = (vrow != nullptr && tok < t_end && tok < kb) ? __ldg(vrow + tok) : -1;
    }
  };
  // checks the positions of the block at t0 and issues its page-table loads
  auto load_pages = [&](int t0, int* p, int* pg) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int tok = t0 + 32 * q4 + lane;
      int pos = -1;
      if (tok < t_end) {
        if (tok < kb) {
          pos = vrow ? p[q4] : tok;
          if (pos < 0 || pos >= nv) { flag_status(status, kStatusBadIndex); pos = -1; }
        } else {
          pos = nv + (tok - kb);
        }
      }
      p[q4] = pos;
      pg[q4] = pos >= 0 ? __ldg(bt + (pos >> 4)) : -1;
    }
  };
  auto form_rows = [&](const int* p, const int* pg, uint32_t* r) {
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint32_t rid = kNoRowM;
      if (p[q4] >= 0) {
        const int page = pg[q4];
        if (page >= 0 && page < num_blocks)
          rid = append && p[q4] == nv + nt ? kNewRowId
                                           : (((uint32_t)page * (uint32_t)Hkv + (uint32_t)g) << 4) | (uint32_t)(p[q4] & 15);
        else
          flag_status(status, kStatusBadBlock);
      }
      r[q4] = rid;
    }
  };
  // row ids of sub-tile i (16 tokens): lanes 0..15 hold them afterwards
  auto rows_of = [&](int i) -> uint32_t {
    const int q4 = (i >> 1) & 3;
    const uint32_t v = q4 == 0 ? blk_cur[0] : q4 == 1 ? blk_cur[1] : q4 == 2 ? blk_cur[2] : blk_cur[3];
    return __shfl_sync(0xffffffffu, v, (lane & 15) + 16 * (i & 1));
  };
  {
    int pos0[4], pg0[4];
    load_idx(t_begin, pos0);
    if (nsub > 8) load_idx(t_begin + 128, pos_a);
    if (nsub > 16) load_idx(t_begin + 256, pos_b);
    load_pages(t_begin, pos0, pg0);
    if (nsub > 8) load_pages(t_begin + 128, pos_a, pg_a);
    form_rows(pos0, pg0, blk_cur);
  }
#pragma unroll
  for (int s = 0; s < kMmaStages - 1; ++s) {
    if (s < nsub) rows[s] = issue(t_begin + s * kSubTile, s, rows_of(s));
    else cp_async_commit();
  }
  // ldmatrix row addresses: lane -> (matrix mi = lane / 8, row ri = lane % 8)
  const int mi = lane >> 3, ri = lane & 7;
  for (int it = 0; it < nsub; ++it) {
    const int s = it % kMmaStages;
    const int nxt = it + kMmaStages - 1;
    if (nxt < nsub) {
      if ((nxt & 7) == 0) {       // first sub-tile of a new 128-token block
        form_rows(pos_a, pg_a, blk_cur);
        if (nxt + 8 < nsub) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) pos_a[q4] = pos_b[q4];
          load_pages(t_begin + (nxt + 8) * kSubTile, pos_a, pg_a);
        }
        if (nxt + 16 < nsub) load_idx(t_begin + (nxt + 16) * kSubTile, pos_b);
      }
      rows[nxt % kMmaStages] = issue(t_begin + nxt * kSubTile, nxt % kMmaStages, rows_of(nxt));
    } else {
      cp_async_commit();
    }
    cp_async_wait<kMmaStages - 1>();
    __syncwarp();
    const uint32_t kbase = smem_u32(my + (size_t)s * 2 * TILE_BYTES);
    const uint32_t vbase = kbase + TILE_BYTES;

    // S = Q K^T over 16 tokens: two n-tiles (tokens 0-7, 8-15)
    float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      // matrices: (tok 0-7, dims 16ks..+7), (tok 0-7, +8..+15), (tok 8-15, ..), (tok 8-15, ..)
      const int tok = (mi >> 1) * 8 + ri;
      const int c = ks * 2 + (mi & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kbase + tok * D * 2 + ((c ^ (tok & 7)) * 16), b0, b1, b2, b3);
      mma_bf16_16816(sacc[0], qa[ks], b0, b1);
      mma_bf16_16816(sacc[1], qa[ks], b2, b3);
    }
    // mask tokens that are outside the split or unresolved
    const uint32_t rid = rows[s];
    const int tc = (lane & 3) * 2;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool valid = __shfl_sync(0xffffffffu, rid, nt * 8 + tc + e) != kNoRowM;
        sacc[nt][e] = valid ? sacc[nt][e] * scale_log2 : -INFINITY;
        sacc[nt][2 + e] = valid ? sacc[nt][2 + e] * scale_log2 : -INFINITY;
      }
    // online softmax, rows r (h = 0) and r + 8 (h = 1)
    float alpha[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      float mx = fmaxf(fmaxf(sacc[0][2 * hh], sacc[0][2 * hh + 1]), fmaxf(sacc[1][2 * hh], sacc[1][2 * hh + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float mn = fmaxf(m_r[hh], mx);
      if (mn == -INFINITY) {
        alpha[hh] = 1.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) sacc[nt][2 * hh] = sacc[nt][2 * hh + 1] = 0.f;
      } else {
        alpha[hh] = fast_exp2(m_r[hh] - mn);
        float ls = 0.f;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float p = fast_exp2(sacc[nt][2 * hh + e] - mn);
            sacc[nt][2 * hh + e] = p;
            ls += p;
          }
        l_r[hh] = l_r[hh] * alpha[hh] + ls;
        m_r[hh] = mn;
      }
    }
#pragma unroll
    for (int j = 0; j < NT_O; ++j) {
      o[j][0] *= alpha[0];
      o[j][1] *= alpha[0];
      o[j][2] *= alpha[1];
      o[j][3] *= alpha[1];
    }
    // P (16 heads x 16 tokens) as the bf16 A operand
    uint32_t pa[4];
    pa[0] = pack_bf16(sacc[0][0], sacc[0][1]);
    pa[1] = pack_bf16(sacc[0][2], sacc[0][3]);
    pa[2] = pack_bf16(sacc[1][0], sacc[1][1]);
    pa[3] = pack_bf16(sacc[1][2], sacc[1][3]);
    // O += P V: per ldmatrix.x4.trans two output n-tiles (16 dims)
#pragma unroll
    for (int j2 = 0; j2 < NT_O / 2; ++j2) {
      // matrices: (tok 0-7, dims 16j2..+7), (tok 8-15, same), (tok 0-7, +8..), (tok 8-15, +8..)
      const int tok = (mi & 1) * 8 + ri;
      const int c = j2 * 2 + (mi >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vbase + tok * D * 2 + ((c ^ (tok & 7)) * 16), b0, b1, b2, b3);
      mma_bf16_16816(o[2 * j2], pa, b0, b1);
      mma_bf16_16816(o[2 * j2 + 1], pa, b2, b3);
    }
    __syncwarp();
  }
  cp_async_wait<0>();

  // row sums over the 4 lanes of a row, then this split's partials
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    l_r[hh] += __shfl_xor_sync(0xffffffffu, l_r[hh], 1);
    l_r[hh] += __shfl_xor_sync(0xffffffffu, l_r[hh], 2);
  }
  const size_t pi = ((size_t)bg * nsplit + split) * G;
  const int r0 = lane >> 2;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    const int hrow = r0 + 8 * hh;
    if (hrow < G) {
#pragma unroll
      for (int j = 0; j < NT_O; ++j)
        *reinterpret_cast<float2*>(part_o + (pi + hrow) * D + j * 8 + (lane & 3) * 2) =
            make_float2(o[j][2 * hh], o[j][2 * hh + 1]);
      if ((lane & 3) == 0) {
        part_ml[(pi + hrow) * 2] = m_r[hh];
        part_ml[(pi + hrow) * 2 + 1] = l_r[hh];
      }
    }
  }

  // the last warp to finish this (sequence, KV head) merges every split
  if (split_done == nullptr) return;
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(split_done + bg, 1) == nsplit - 1;
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  constexpr int DPL = D / 32;
  const size_t base = (size_t)bg * nsplit;
  for (int hh = 0; hh < G; ++hh) {
    float M = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, __ldcg(part_ml + ((base + s) * G + hh) * 2));
    M = warp_max(M);
    float L = 0.f, acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const size_t ps = (base + s) * G + hh;
      const float ms = __ldcg(part_ml + ps * 2);
      const float wgt = (ms == -INFINITY) ? 0.f : fast_exp2(ms - M);
      L = fmaf(wgt, __ldcg(part_ml + ps * 2 + 1), L);
      const float* po = part_o + ps * D + lane * DPL;
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[e] = fmaf(wgt, __ldcg(po + e), acc[e]);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint16_t* dst = out + ((size_t)b * H + g * G + hh) * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; ++e) dst[e] = (uint16_t)f32_to_bf16_bits(acc[e] * inv);
    if (lse != nullptr && lane == 0)
      lse[(size_t)b * H + g * G + hh] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
  if (lane == 0) split_done[bg] = 0;
}

size_t attn_mma_smem_bytes(int D) { return (size_t)kMmaWarps * kMmaStages * 2 * kSubTile * D * 2; }

cudaError_t launch_sparse_attn_mma(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream) {
  const long long warps = (long long)a.batch * a.Hkv * p.nsplit;
  const unsigned grid = (unsigned)((warps + kMmaWarps - 1) / kMmaWarps);
  const size_t smem = attn_mma_smem_bytes(a.D);
  const int G = a.H / a.Hkv;
  // the instantiation for this call: head dim and whether it appends a token
  const bool app = a.k_new != nullptr;
  auto kernel = a.D == 128 ? (app ? sparse_attn_mma_kernel<128, true> : sparse_attn_mma_kernel<128, false>)
                           : (app ? sparse_attn_mma_kernel<64, true> : sparse_attn_mma_kernel<64, false>);
  static bool attr_set[64][4] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int di = (a.D == 128 ? 1 : 0) + (app ? 2 : 0);
  if (dev < 0 || dev >= 64 || !attr_set[dev][di]) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_set[dev][di] = true;
  }
#define SV_MMA_ARGS                                                                                        \
  static_cast<const uint16_t*>(a.q), a.H, G, static_cast<const uint16_t*>(a.k_pool),                        \
      static_cast<const uint16_t*>(a.v_pool), a.num_blocks, a.Hkv, a.block_table, a.max_blocks, a.vis_idx, \
      a.k_vis, a.n_vis, a.n_text, a.scale * kLog2e, a.batch, p.nsplit, p.chunk, a.part_ml, a.part_o,       \
      a.status, a.split_done, static_cast<uint16_t*>(a.out), a.lse, a.lens,                                \
      static_cast<const uint16_t*>(a.k_new), static_cast<const uint16_t*>(a.v_new),                         \
      static_cast<uint16_t*>(const_cast<void*>(a.k_pool)), static_cast<uint16_t*>(const_cast<void*>(a.v_pool))
  e = launch_dependent(kernel, dim3(grid), dim3(kMmaWarps * 32), smem, stream, SV_MMA_ARGS);
#undef SV_MMA_ARGS
  return e;
}

}  // namespace sv
