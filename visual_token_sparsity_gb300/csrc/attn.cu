// Sparse decode attention over the retrieved visual tokens plus all text
// tokens, gathered from the paged bf16 cache.
//
// velog.io SparseVILA summary §3.2 (decode is memory-bound: read only the
// query-relevant subset of the preserved visual cache) and §4.5 kernel table
// ("decoding attention" over the reduced KV).  For query head h of KV group
// g = h / G the token set is T = vis_idx[b][g] U text, and
//   out = sum_{t in T} softmax_t(scale q.k_t) v_t
// with an fp32 online softmax in the log2 domain.
//
// Split-K: every warp owns one (sequence, KV head, token split) and streams
// its tokens in tiles.  Per tile each lane looks up one token's page through
// the block table, the warp issues all K and V row loads (16 B per lane, whole
// 128/256-byte rows per lane group) and then folds the per-lane partial dot
// products with a butterfly reduce-scatter.  The G query heads of the group
// share every K/V load.  Per-split (m, l, o) partials go to the workspace; the
// last warp to finish a (sequence, KV head) -- a device-scope counter, no
// waiting -- merges them and writes the bf16 output and the lse.
#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {

template <int D, int G>
struct AttnShape {
  static constexpr int LPT = D / 8;
  static constexpr int TPI = 32 / LPT;
  static constexpr int TILE = G <= 2 ? 32 : (G <= 4 ? 16 : 8);
  static constexpr int NL = TILE / TPI;
  static constexpr int DUP = LPT / NL;
};

constexpr int kAttnWarps = 4;
constexpr int kAttnTargetWarps = 4096;
constexpr int kAttnMaxSplits = 1024;
constexpr uint32_t kNoRow = 0xffffffffu;

int attn_tile(int G) { return G <= 2 ? 32 : (G <= 4 ? 16 : 8); }

}  // namespace

AttnPlan attn_plan(int B, int Hkv, int G, int n_tokens) {
  AttnPlan p;
  p.tile = attn_tile(G);
  const int tiles = (n_tokens + p.tile - 1) / p.tile;
  const long long units = (long long)B * Hkv;
  long long tiles_total = units * (tiles > 0 ? tiles : 1);
  long long tpw = (tiles_total + kAttnTargetWarps - 1) / kAttnTargetWarps;
  if (tpw < 1) tpw = 1;
  long long min_tpw = (tiles + kAttnMaxSplits - 1) / kAttnMaxSplits;
  if (tpw < min_tpw) tpw = min_tpw;
  p.chunk = (int)(tpw * p.tile);
  p.nsplit = n_tokens > 0 ? (n_tokens + p.chunk - 1) / p.chunk : 1;
  // nsplit <= ceil(tiles / tpw) <= min(tiles, ceil(target / units), max): a
  // bound that never decreases as n_tokens grows (workspace sizing).
  long long ub = tiles > 0 ? tiles : 1;
  const long long per_unit = (kAttnTargetWarps + units - 1) / (units > 0 ? units : 1);
  if (ub > per_unit) ub = per_unit;
  if (ub > kAttnMaxSplits) ub = kAttnMaxSplits;
  p.nsplit_max = (int)(ub > p.nsplit ? ub : p.nsplit);
  return p;
}

template <int D, int G>
__global__ void __launch_bounds__(kAttnWarps * 32, (G == 1 ? 3 : 1))
sparse_attn_split_kernel(const uint16_t* __restrict__ q, int H,
                         const uint16_t* __restrict__ k_pool, const uint16_t* __restrict__ v_pool,
                         int num_blocks, int Hkv, const int32_t* __restrict__ block_table,
                         int max_blocks, const int32_t* __restrict__ vis_idx, int k_vis,
                         int n_vis, int n_text, float scale_log2, int batch, int nsplit, int chunk,
                         float* __restrict__ part_ml, float* __restrict__ part_o, int* status,
                         int* split_done, uint16_t* __restrict__ out, float* __restrict__ lse) {
  using S = AttnShape<D, G>;
  constexpr int LPT = S::LPT, TPI = S::TPI, TILE = S::TILE, NL = S::NL, DUP = S::DUP;

  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * kAttnWarps + (threadIdx.x >> 5);
  if (w >= (long long)batch * Hkv * nsplit) return;
  const int split = (int)(w % nsplit);
  const int bg = (int)(w / nsplit);
  const int b = bg / Hkv, g = bg % Hkv;
  const int T = k_vis + n_text;
  const int t_begin = split * chunk;
  const int t_end = min(T, t_begin + chunk);
  const int dim0 = (lane % LPT) * 8;

  float qv[G][8];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    const uint4 u = *reinterpret_cast<const uint4*>(q + ((size_t)b * H + g * G + hh) * D + dim0);
    const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      qv[hh][2 * c] = bf16_lo(wv[c]) * scale_log2;
      qv[hh][2 * c + 1] = bf16_hi(wv[c]) * scale_log2;
    }
  }

  float m[G], lsum[G], o[G][8];
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
    m[hh] = -INFINITY;
    lsum[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) o[hh][e] = 0.f;
  }

  const int32_t* bt = block_table + (size_t)b * max_blocks;
  const int32_t* vrow = vis_idx ? vis_idx + (size_t)bg * k_vis : nullptr;
  const int my_slot = (lane % LPT) / DUP;              // value index after the fold
  const int my_tok = my_slot * TPI + lane / LPT;       // token of the tile held after the fold

  for (int t0 = t_begin; t0 < t_end; t0 += TILE) {
    uint32_t rowid = kNoRow;
    const int tok = t0 + lane;
    if (lane < TILE && tok < t_end) {
      int pos;
      if (tok < k_vis) {
        pos = vrow ? __ldg(vrow + tok) : tok;
        if (pos < 0 || pos >= n_vis) { flag_status(status, kStatusBadIndex); pos = -1; }
      } else {
        pos = n_vis + (tok - k_vis);
      }
      if (pos >= 0) {
        const int page = __ldg(bt + (pos >> 4));
        if (page >= 0 && page < num_blocks)
          rowid = (((uint32_t)page * (uint32_t)Hkv + (uint32_t)g) << 4) | (uint32_t)(pos & 15);
        else
          flag_status(status, kStatusBadBlock);
      }
    }

    uint4 kd[NL], vd[NL];
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const uint32_t r = __shfl_sync(0xffffffffu, rowid, i * TPI + lane / LPT);
      if (r != kNoRow) {
        kd[i] = ld_stream16(k_pool + (size_t)r * D + dim0);
        vd[i] = ld_stream16(v_pool + (size_t)r * D + dim0);
      } else {
        kd[i] = make_uint4(0, 0, 0, 0);
        vd[i] = make_uint4(0, 0, 0, 0);
      }
    }
    const bool mine_valid = __shfl_sync(0xffffffffu, rowid, my_tok) != kNoRow;

    float p[G];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float part[NL];
#pragma unroll
      for (int i = 0; i < NL; ++i) {
        const uint32_t wv[4] = {kd[i].x, kd[i].y, kd[i].z, kd[i].w};
        float a = 0.f;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          a = fmaf(qv[hh][2 * c], bf16_lo(wv[c]), a);
          a = fmaf(qv[hh][2 * c + 1], bf16_hi(wv[c]), a);
        }
        part[i] = a;
      }
      GroupReduce<NL, LPT>::run(part, lane);
      const float s = mine_valid ? part[0] : -INFINITY;
      const float m_new = fmaxf(m[hh], warp_max(s));
      float alpha, pj;
      if (m_new == -INFINITY) {
        alpha = 1.f;
        pj = 0.f;
      } else {
        alpha = fast_exp2(m[hh] - m_new);
        pj = fast_exp2(s - m_new);
      }
      m[hh] = m_new;
      lsum[hh] = lsum[hh] * alpha + ((lane % DUP) == 0 ? pj : 0.f);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[hh][e] *= alpha;
      p[hh] = pj;
    }

#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const int src = (lane / LPT) * LPT + i * DUP;
      const uint32_t wv[4] = {vd[i].x, vd[i].y, vd[i].z, vd[i].w};
      float v[8];
#pragma unroll
      for (int c = 0; c < 4; ++c) { v[2 * c] = bf16_lo(wv[c]); v[2 * c + 1] = bf16_hi(wv[c]); }
#pragma unroll
      for (int hh = 0; hh < G; ++hh) {
        const float pj = __shfl_sync(0xffffffffu, p[hh], src);
#pragma unroll
        for (int e = 0; e < 8; ++e) o[hh][e] = fmaf(pj, v[e], o[hh][e]);
      }
    }
  }

  // fold the TPI lane groups and the per-lane softmax sums
#pragma unroll
  for (int hh = 0; hh < G; ++hh) {
#pragma unroll
    for (int mk = LPT; mk < 32; mk <<= 1)
#pragma unroll
      for (int e = 0; e < 8; ++e) o[hh][e] += __shfl_xor_sync(0xffffffffu, o[hh][e], mk);
    lsum[hh] = warp_sum(lsum[hh]);
  }
  const size_t pi = ((size_t)bg * nsplit + split) * G;
  if (lane < LPT) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      float4* dst = reinterpret_cast<float4*>(part_o + (pi + hh) * D + dim0);
      dst[0] = make_float4(o[hh][0], o[hh][1], o[hh][2], o[hh][3]);
      dst[1] = make_float4(o[hh][4], o[hh][5], o[hh][6], o[hh][7]);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
      part_ml[(pi + hh) * 2] = m[hh];
      part_ml[(pi + hh) * 2 + 1] = lsum[hh];
    }
  }

  // The last warp to finish this (sequence, KV head) merges every split:
  // out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s, M = max_s m_s.
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(split_done + bg, 1) == nsplit - 1;
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  constexpr int DPL = D / 32;   // output dims per lane
  const size_t base = (size_t)bg * nsplit;
  for (int hh = 0; hh < G; ++hh) {
    float M = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, __ldcg(part_ml + ((base + s) * G + hh) * 2));
    M = warp_max(M);
    float L = 0.f, acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
#pragma unroll 4
    for (int s = 0; s < nsplit; ++s) {
      const size_t ps = (base + s) * G + hh;
      const float ms = __ldcg(part_ml + ps * 2);
      const float w = (ms == -INFINITY) ? 0.f : fast_exp2(ms - M);
      L = fmaf(w, __ldcg(part_ml + ps * 2 + 1), L);
      const float* po = part_o + ps * D + lane * DPL;
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[e] = fmaf(w, __ldcg(po + e), acc[e]);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint16_t* dst = out + ((size_t)b * H + g * G + hh) * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; ++e) dst[e] = (uint16_t)f32_to_bf16_bits(acc[e] * inv);
    if (lse != nullptr && lane == 0)
      lse[(size_t)b * H + g * G + hh] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
  }
  if (lane == 0) split_done[bg] = 0;   // ready for the next call
}

template <int D, int G>
static void launch_split(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream) {
  const long long warps = (long long)a.batch * a.Hkv * p.nsplit;
  const unsigned grid = (unsigned)((warps + kAttnWarps - 1) / kAttnWarps);
  sparse_attn_split_kernel<D, G><<<grid, kAttnWarps * 32, 0, stream>>>(
      static_cast<const uint16_t*>(a.q), a.H, static_cast<const uint16_t*>(a.k_pool),
      static_cast<const uint16_t*>(a.v_pool), a.num_blocks, a.Hkv, a.block_table, a.max_blocks,
      a.vis_idx, a.k_vis, a.n_vis, a.n_text, a.scale * kLog2e, a.batch, p.nsplit, p.chunk,
      a.part_ml, a.part_o, a.status, a.split_done, static_cast<uint16_t*>(a.out), a.lse);
}

template <int D>
static bool dispatch_g(const AttnArgs& a, const AttnPlan& p, cudaStream_t s) {
  switch (a.H / a.Hkv) {
    case 1: launch_split<D, 1>(a, p, s); return true;
    case 2: launch_split<D, 2>(a, p, s); return true;
    case 3: launch_split<D, 3>(a, p, s); return true;
    case 4: launch_split<D, 4>(a, p, s); return true;
    case 5: launch_split<D, 5>(a, p, s); return true;
    case 6: launch_split<D, 6>(a, p, s); return true;
    case 7: launch_split<D, 7>(a, p, s); return true;
    case 8: launch_split<D, 8>(a, p, s); return true;
    default: return false;
  }
}

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream) {
  const int G = a.H / a.Hkv;
  const AttnPlan p = attn_plan(a.batch, a.Hkv, G, a.k_vis + a.n_text);
  const bool ok = a.D == 128 ? dispatch_g<128>(a, p, stream) : dispatch_g<64>(a, p, stream);
  if (!ok) return cudaErrorInvalidValue;
  return cudaGetLastError();
}
}  // namespace sv
