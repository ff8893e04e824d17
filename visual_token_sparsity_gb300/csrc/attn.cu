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
// This file holds the CUDA-core kernel used for G <= 2 query heads per KV
// head; attn_mma.cu holds the tensor-core kernel for larger groups.
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

#ifndef SV_ATTN_TILE
#define SV_ATTN_TILE 8         // tokens per warp step of the G <= 2 kernel (large batches)
#endif
#ifndef SV_ATTN_SMALL_UNITS
#define SV_ATTN_SMALL_UNITS 8  // at most this many (sequence, KV head) units: 32-token steps
#endif
#ifndef SV_ATTN_MMA_MIN_G
#define SV_ATTN_MMA_MIN_G 3    // groups of at least this many heads use the tensor-core kernel
#endif
#ifndef SV_ATTN_MIN_BLOCKS
#define SV_ATTN_MIN_BLOCKS 7   // resident CTAs per SM the G = 1, 8-token kernel is register-capped for
#endif

namespace sv {

namespace {

template <int D, int G, int TILE_ = SV_ATTN_TILE>
struct AttnShape {
  static constexpr int LPT = D / 8;
  static constexpr int TPI = 32 / LPT;
  static constexpr int TILE = G <= 2 ? TILE_ : (G <= 4 ? 16 : 8);
  static constexpr int NL = TILE / TPI;
  static constexpr int DUP = LPT / NL;
};

constexpr int kAttnWarps = 4;
#ifndef SV_ATTN_TARGET_WARPS
#define SV_ATTN_TARGET_WARPS 4096   // <= 152 SMs x 7 CTAs x 4 warps: one wave
#endif
constexpr int kAttnTargetWarps = SV_ATTN_TARGET_WARPS;
// Tensor-core kernel (G >= 3) split plan: at most kMmaTargetWarps warps in
// all (152 SMs x 4 CTAs x 2 warps resident: one wave), at least
// kMmaMinTokens tokens and at most kMmaMaxSplits splits per (sequence, KV
// head): short calls gain from many short splits, while above ~200 splits
// the merge kernel's per-split loads cost more than the extra warps save.
#ifndef SV_MMA_TARGET_WARPS
#define SV_MMA_TARGET_WARPS 1216
#endif
#ifndef SV_MMA_MIN_TOKENS
#define SV_MMA_MIN_TOKENS 32
#endif
#ifndef SV_MMA_MAX_SPLITS
#define SV_MMA_MAX_SPLITS 200
#endif
constexpr int kMmaTargetWarps = SV_MMA_TARGET_WARPS;
constexpr int kMmaMinTokens = SV_MMA_MIN_TOKENS;
constexpr int kMmaMaxSplits = SV_MMA_MAX_SPLITS;
constexpr int kAttnMaxSplits = 1024;
constexpr int kFusedMergeMaxSplits = 32;   // above this a separate merge kernel runs
#ifndef SV_MMA_FUSED_MAX
#define SV_MMA_FUSED_MAX 0
#endif
// Tensor-core kernel: its last warp would merge G heads x nsplit partial rows
// one after another, which measured slower than the merge kernel at every
// size tried (G 7 with 7-28 splits: 31.4 against 22.3 us for 16 sequences of
// 1568 tokens), so by default (a product bound of 0) that path always runs
// the merge kernel.
constexpr int kMmaFusedMergeMax = SV_MMA_FUSED_MAX;
constexpr uint32_t kNoRow = kNoRowId;

// tokens per warp step: one 16-token MMA sub-tile for the tensor-core kernel
// (attn_mma.cu, G >= 3); for the CUDA-core kernel (G <= 2) 8-token steps at
// 7 CTAs per SM when the batch fills the GPU, and 32-token steps for a few
// (sequence, KV head) units, where fewer splits shorten the serial merge of
// a latency-bound call
bool attn_uses_mma(int G) { return G >= SV_ATTN_MMA_MIN_G; }
int attn_tile(int G, long long units) {
  if (attn_uses_mma(G)) return 16;
  return units <= SV_ATTN_SMALL_UNITS ? 32 : SV_ATTN_TILE;
}

}  // namespace

AttnPlan attn_plan(int B, int Hkv, int G, int n_tokens) {
  AttnPlan p;
  const long long units = (long long)B * Hkv;
  p.tile = attn_tile(G, units);
  const int tiles = (n_tokens + p.tile - 1) / p.tile;
  long long tiles_total = units * (tiles > 0 ? tiles : 1);
  long long tpw;
  if (attn_uses_mma(G)) {
    long long cap = kMmaTargetWarps / (units > 0 ? units : 1);
    if (cap > kMmaMaxSplits) cap = kMmaMaxSplits;
    if (cap < 1) cap = 1;
    tpw = ((tiles > 0 ? tiles : 1) + cap - 1) / cap;
    const long long min_tpw = (kMmaMinTokens + p.tile - 1) / p.tile;
    if (tpw < min_tpw) tpw = min_tpw;
  } else {
    tpw = (tiles_total + kAttnTargetWarps - 1) / kAttnTargetWarps;
    if (tpw < 1) tpw = 1;
    const long long min_tpw = (tiles + kAttnMaxSplits - 1) / kAttnMaxSplits;
    if (tpw < min_tpw) tpw = min_tpw;
  }
  // CUDA-core path: stay within the fused merge (at most kFusedMergeMaxSplits
  // splits, merged by the last warp) when that still leaves 512 or more warps;
  // a separate merge launch costs more than longer splits at small batches
  if (!attn_uses_mma(G) && (tiles + tpw - 1) / tpw > kFusedMergeMaxSplits) {
    const long long tpw2 = (tiles + kFusedMergeMaxSplits - 1) / kFusedMergeMaxSplits;
    if (units * ((tiles + tpw2 - 1) / tpw2) >= 512) tpw = tpw2;
  }
  p.chunk = (int)(tpw * p.tile);
  p.nsplit = n_tokens > 0 ? (n_tokens + p.chunk - 1) / p.chunk : 1;
  // nsplit <= ceil(tiles / tpw) <= min(tiles, ceil(target / units), max): a
  // bound that never decreases as n_tokens grows (workspace sizing).
  // chunk >= max(tile, min_tokens), so nsplit <= ceil(n_tokens / that)
  const long long min_chunk =
      attn_uses_mma(G) && kMmaMinTokens > p.tile ? (kMmaMinTokens + p.tile - 1) / p.tile * p.tile : p.tile;
  long long ub = (n_tokens + min_chunk - 1) / min_chunk;
  if (ub < 1) ub = 1;
  const long long target = attn_uses_mma(G) ? kMmaTargetWarps : kAttnTargetWarps;
  const long long per_unit = (target + units - 1) / (units > 0 ? units : 1);
  if (ub > per_unit) ub = per_unit;
  if (ub > kAttnMaxSplits) ub = kAttnMaxSplits;
  if (attn_uses_mma(G) && ub > kMmaMaxSplits) ub = kMmaMaxSplits;
  p.nsplit_max = (int)(ub > p.nsplit ? ub : p.nsplit);
  return p;
}

static bool attn_fused_merge(const AttnPlan& p, int G) {
  if (p.nsplit > kFusedMergeMaxSplits) return false;
  return !attn_uses_mma(G) || (long long)G * p.nsplit <= kMmaFusedMergeMax;
}

int attn_kernel_count(int B, int Hkv, int G, int n_tokens) {
  return attn_fused_merge(attn_plan(B, Hkv, G, n_tokens), G) ? 1 : 2;
}

// APPEND: the fused append-and-attend variant (k_new / v_new set); a separate
// instantiation, so that the plain call's hot loop carries none of it.
template <int D, int G, int TILE_, bool APPEND>
__global__ void __launch_bounds__(kAttnWarps * 32, (G == 1 ? (TILE_ <= 8 ? SV_ATTN_MIN_BLOCKS : 3) : 1))
sparse_attn_split_kernel(const uint16_t* __restrict__ q, int H,
                         const uint16_t* __restrict__ k_pool, const uint16_t* __restrict__ v_pool,
                         int num_blocks, int Hkv, const int32_t* __restrict__ block_table,
                         int max_blocks, const int32_t* __restrict__ vis_idx, int k_vis,
                         int n_vis, int n_text, float scale_log2, int batch, int nsplit, int chunk,
                         float* __restrict__ part_ml, float* __restrict__ part_o, int* status,
                         int* split_done, uint16_t* __restrict__ out, float* __restrict__ lse,
                         SeqLens lens, const uint16_t* __restrict__ k_new, const uint16_t* __restrict__ v_new,
                         uint16_t* k_store, uint16_t* v_store) {
  using S = AttnShape<D, G, TILE_>;
  constexpr int LPT = S::LPT, TPI = S::TPI, TILE = S::TILE, NL = S::NL, DUP = S::DUP;

  grid_dep_sync();
  const int lane = threadIdx.x & 31;
  const long long w = (long long)blockIdx.x * kAttnWarps + (threadIdx.x >> 5);
  if (w >= (long long)batch * Hkv * nsplit) return;
  const int split = (int)(w % nsplit);
  const int bg = (int)(w / nsplit);
  const int b = bg / Hkv, g = bg % Hkv;
  // this sequence's counts (k_vis, n_vis, n_text are capacities with
  // per-sequence lengths; splits past its tokens stay empty)
  int nv, nt, kb;
  const bool seq_ok = attn_lengths(lens, vis_idx != nullptr, b, n_vis, n_text, k_vis,
                                   lane == 0 && split == 0 && g == 0, status, nv, nt, kb);
  // a fused append adds the new token (cache position nv + nt) as the last one
  const bool append = APPEND && seq_ok;
  const int T = kb + nt + (append ? 1 : 0);
  const int t_begin = split * chunk;
  const int t_end = min(T, t_begin + chunk);
  const int dim0 = (lane % LPT) * 8;
  if (append && split == 0)
    store_new_token(k_store, v_store, k_new, v_new, block_table + (size_t)b * max_blocks, num_blocks, Hkv, D, b, g,
                    nv + nt, lane);

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

  // Token -> pool row id for the TILE tokens starting at t0 (lane < TILE), as
  // a 2-stage software pipeline: a tile's visual indices are loaded two tiles
  // ahead and its page-table entries one tile ahead, so no load's latency
  // falls inside the iteration that needs it.
  auto load_pos = [&](int t0) -> int {
    const int tok = t0 + lane;
    if (lane >= TILE || tok >= t_end) return -1;
    if (tok >= kb) return nv + (tok - kb);
    const int pos = vrow ? __ldg(vrow + tok) : tok;
    if (pos < 0 || pos >= nv) { flag_status(status, kStatusBadIndex); return -1; }
    return pos;
  };
  auto lookup = [&](int pos) -> uint32_t {
    if (pos < 0) return kNoRow;
    const int page = __ldg(bt + (pos >> 4));
    if (page >= 0 && page < num_blocks) {
      if (append && pos == nv + nt) return kNewRowId;   // read from k_new / v_new
      return (((uint32_t)page * (uint32_t)Hkv + (uint32_t)g) << 4) | (uint32_t)(pos & 15);
    }
    flag_status(status, kStatusBadBlock);
    return kNoRow;
  };
  // the TILE tokens' K and V rows for this lane (16 bytes each)
  auto issue = [&](uint32_t rowid, uint4* kd, uint4* vd) {
#pragma unroll
    for (int i = 0; i < NL; ++i) {
      const uint32_t r = __shfl_sync(0xffffffffu, rowid, i * TPI + lane / LPT);
      if (r != kNoRow) {
        const bool fresh = APPEND && r == kNewRowId;
        kd[i] = ld_stream16((fresh ? k_new + (size_t)bg * D : k_pool + (size_t)r * D) + dim0);
        vd[i] = ld_stream16((fresh ? v_new + (size_t)bg * D : v_pool + (size_t)r * D) + dim0);
      } else {
        kd[i] = make_uint4(0, 0, 0, 0);
        vd[i] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  // scores, online softmax and P.V of one tile
  auto consume = [&](uint32_t rowid, const uint4* kd, const uint4* vd) {
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
  };

  uint32_t next_rowid = lookup(load_pos(t_begin));
  int pos_ahead = load_pos(t_begin + TILE);
  for (int t0 = t_begin; t0 < t_end; t0 += TILE) {
    const uint32_t rowid = next_rowid;
    uint4 kd[NL], vd[NL];
    issue(rowid, kd, vd);
    next_rowid = lookup(pos_ahead);
    pos_ahead = load_pos(t0 + 2 * TILE);
    consume(rowid, kd, vd);
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
  // (With many splits a separate merge kernel does this instead.)
  if (split_done == nullptr) return;
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atomicAdd(split_done + bg, 1) == nsplit - 1;
  if (!__shfl_sync(0xffffffffu, last, 0)) return;
  __threadfence();
  constexpr int DPL = D / 32;   // output dims per lane
  const size_t base = (size_t)bg * nsplit;
  for (int hh = 0; hh < G; ++hh) {
    // lane s holds split s (nsplit <= 32 here): its (m, l) and weight come in
    // one round of loads; the partial rows follow kMergeBatch splits at a time
    float ms = -INFINITY, ls = 0.f;
    if (lane < nsplit) {
      ms = __ldcg(part_ml + ((base + lane) * G + hh) * 2);
      ls = __ldcg(part_ml + ((base + lane) * G + hh) * 2 + 1);
    }
    const float M = warp_max(ms);
    const float w = (ms == -INFINITY) ? 0.f : fast_exp2(ms - M);
    const float L = warp_sum(w * ls);
    float acc[DPL];
#pragma unroll
    for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
    constexpr int kMergeBatch = 8;
    for (int s0 = 0; s0 < nsplit; s0 += kMergeBatch) {
      float x[kMergeBatch][DPL];
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        const float* po = part_o + ((base + s0 + j) * G + hh) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) x[j][e] = s0 + j < nsplit ? __ldcg(po + e) : 0.f;
      }
#pragma unroll
      for (int j = 0; j < kMergeBatch; ++j) {
        const float wj = __shfl_sync(0xffffffffu, w, s0 + j);   // 0 past nsplit
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] = fmaf(wj, x[j][e], acc[e]);
      }
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

template <int D, int G, int TILE>
static cudaError_t launch_split(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream) {
  const long long warps = (long long)a.batch * a.Hkv * p.nsplit;
  const unsigned grid = (unsigned)((warps + kAttnWarps - 1) / kAttnWarps);
  auto kernel = a.k_new != nullptr ? sparse_attn_split_kernel<D, G, TILE, true>
                                   : sparse_attn_split_kernel<D, G, TILE, false>;
  return launch_dependent(kernel, dim3(grid), dim3(kAttnWarps * 32), 0, stream,
                          static_cast<const uint16_t*>(a.q), a.H, static_cast<const uint16_t*>(a.k_pool),
                          static_cast<const uint16_t*>(a.v_pool), a.num_blocks, a.Hkv, a.block_table, a.max_blocks,
                          a.vis_idx, a.k_vis, a.n_vis, a.n_text, a.scale * kLog2e, a.batch, p.nsplit, p.chunk,
                          a.part_ml, a.part_o, a.status, a.split_done, static_cast<uint16_t*>(a.out), a.lse,
                          a.lens, static_cast<const uint16_t*>(a.k_new), static_cast<const uint16_t*>(a.v_new),
                          static_cast<uint16_t*>(const_cast<void*>(a.k_pool)),
                          static_cast<uint16_t*>(const_cast<void*>(a.v_pool)));
}

template <int D, int G>
static cudaError_t launch_split_tile(const AttnArgs& a, const AttnPlan& p, cudaStream_t s) {
  if (p.tile == 32) return launch_split<D, G, 32>(a, p, s);
  return launch_split<D, G, SV_ATTN_TILE>(a, p, s);
}

template <int D>
static cudaError_t dispatch_g(const AttnArgs& a, const AttnPlan& p, cudaStream_t s) {
  switch (a.H / a.Hkv) {
    case 1: return launch_split_tile<D, 1>(a, p, s);
    case 2: return launch_split_tile<D, 2>(a, p, s);
    default: return cudaErrorInvalidValue;
  }
}

// Merges the per-split partials of one (sequence, query head) when there are
// too many splits for the fused single-warp merge.  256 threads: the split
// weights 2^(m_s - M) go to shared memory, then each of the 8 warps sums every
// 8th split (lanes over output dims, 4 splits' loads in flight per lane) and
// the 8 partial vectors are added in shared memory.
__global__ void __launch_bounds__(256)
attn_merge_kernel(const float* __restrict__ part_ml, const float* __restrict__ part_o, int H, int Hkv,
                  int G, int D, int nsplit, uint16_t* __restrict__ out, float* __restrict__ lse) {
  extern __shared__ float wsh[];   // nsplit weights
  __shared__ float red[8];
  __shared__ float4 part[8][32];
  grid_dep_sync();
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh % H;
  const int g = h / G, hh = h % G;
  const size_t base = ((size_t)b * Hkv + g) * nsplit;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float mx = -INFINITY;
  for (int s = tid; s < nsplit; s += blockDim.x) mx = fmaxf(mx, part_ml[((base + s) * G + hh) * 2]);
  mx = warp_max(mx);
  if (lane == 0) red[warp] = mx;
  __syncthreads();
  float M = red[0];
  for (int i = 1; i < 8; ++i) M = fmaxf(M, red[i]);
  __syncthreads();
  float lacc = 0.f;
  for (int s = tid; s < nsplit; s += blockDim.x) {
    const float ms = part_ml[((base + s) * G + hh) * 2];
    const float w = (M == -INFINITY || ms == -INFINITY) ? 0.f : fast_exp2(ms - M);
    wsh[s] = w;
    lacc = fmaf(w, part_ml[((base + s) * G + hh) * 2 + 1], lacc);
  }
  lacc = warp_sum(lacc);
  if (lane == 0) red[warp] = lacc;
  __syncthreads();
  float L = 0.f;
  for (int i = 0; i < 8; ++i) L += red[i];
  const float inv = L > 0.f ? 1.f / L : 0.f;
  // lanes cover the output dims 4 at a time (D = 128: 32 lanes; D = 64: 16 lanes)
  const int nl = D / 4;
  const size_t stride = (size_t)G * D;
  const float* po = part_o + (base * G + hh) * D + lane * 4;
  float4 a0 = make_float4(0.f, 0.f, 0.f, 0.f), a1 = a0;
  if (lane < nl) {
    int s = warp;
    for (; s + 8 < nsplit; s += 16) {
      const float4 x0 = *reinterpret_cast<const float4*>(po + (size_t)s * stride);
      const float4 x1 = *reinterpret_cast<const float4*>(po + (size_t)(s + 8) * stride);
      const float w0 = wsh[s], w1 = wsh[s + 8];
      a0.x = fmaf(w0, x0.x, a0.x); a0.y = fmaf(w0, x0.y, a0.y); a0.z = fmaf(w0, x0.z, a0.z); a0.w = fmaf(w0, x0.w, a0.w);
      a1.x = fmaf(w1, x1.x, a1.x); a1.y = fmaf(w1, x1.y, a1.y); a1.z = fmaf(w1, x1.z, a1.z); a1.w = fmaf(w1, x1.w, a1.w);
    }
    for (; s < nsplit; s += 8) {
      const float4 x0 = *reinterpret_cast<const float4*>(po + (size_t)s * stride);
      const float w0 = wsh[s];
      a0.x = fmaf(w0, x0.x, a0.x); a0.y = fmaf(w0, x0.y, a0.y); a0.z = fmaf(w0, x0.z, a0.z); a0.w = fmaf(w0, x0.w, a0.w);
    }
  }
  part[warp][lane] = make_float4(a0.x + a1.x, a0.y + a1.y, a0.z + a1.z, a0.w + a1.w);
  __syncthreads();
  if (warp == 0 && lane < nl) {
    float4 t = part[0][lane];
    for (int i = 1; i < 8; ++i) {
      const float4 u = part[i][lane];
      t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
    }
    uint16_t* dst = out + (size_t)bh * D + lane * 4;
    dst[0] = (uint16_t)f32_to_bf16_bits(t.x * inv);
    dst[1] = (uint16_t)f32_to_bf16_bits(t.y * inv);
    dst[2] = (uint16_t)f32_to_bf16_bits(t.z * inv);
    dst[3] = (uint16_t)f32_to_bf16_bits(t.w * inv);
  }
  if (lse != nullptr && tid == 0) lse[bh] = L > 0.f ? (M + log2f(L)) * 0.6931471805599453f : -INFINITY;
}

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream) {
  const int G = a.H / a.Hkv;
  // a fused append attends one token more
  const AttnPlan p = attn_plan(a.batch, a.Hkv, G, a.k_vis + a.n_text + (a.k_new != nullptr ? 1 : 0));
  AttnArgs b = a;
  const bool fused_merge = attn_fused_merge(p, G);
  if (!fused_merge) b.split_done = nullptr;
  cudaError_t e;
  if (attn_uses_mma(G)) {
    e = launch_sparse_attn_mma(b, p, stream);
  } else {
    e = a.D == 128 ? dispatch_g<128>(b, p, stream) : dispatch_g<64>(b, p, stream);
  }
  if (e != cudaSuccess || fused_merge) return e;
  return launch_dependent(attn_merge_kernel, dim3(a.batch * a.H), dim3(256), (size_t)p.nsplit * sizeof(float),
                          stream, a.part_ml, a.part_o, a.H, a.Hkv, G, a.D, p.nsplit, static_cast<uint16_t*>(a.out),
                          a.lse);
}
}  // namespace sv
