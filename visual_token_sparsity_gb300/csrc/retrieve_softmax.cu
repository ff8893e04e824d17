// Softmax-normalised query-aware retrieval.
//
// velog.io SparseVILA summary §3.2 "Query-Aware Token Selection": the
// aggregated attention strength between the question's rows and the cached
// vision tokens ranks the tokens; the pages' retrieval kernel runs alongside
// the question's FlashAttention-2 prefill.  Here the strength of visual token
// j for KV head g is the attention probability mass it receives,
//   score[b][g][j] = sum_{r<R} sum_{h in g} exp(scale q_{r,h}.k_j - lse_{r,h}),
// with lse_{r,h} the row's log-sum-exp over every cached token (pass 1), or a
// caller's own prefill statistics when given (the fused form: no pass 1).
//
// The R x G question rows of one (sequence, KV head) are a small matrix, so
// the logits are warp-level tensor-core tiles (mma.sync m16n8k16, rows padded
// to 16): each CTA stages its unit's question rows in XOR-swizzled shared
// memory once; each warp streams 16-token K sub-tiles of its token range
// through a 2-stage cp.async ring, keeps the sub-tile's K fragments in
// registers and loops over the 16-row query tiles.  Pass 1 keeps per-row
// online (max, sum) partials that a small kernel merges; pass 2 sums
// exp2(z - lse) over the rows of every query tile into per-token scores in a
// fixed order (deterministic).  The top-k is the row top-k used elsewhere.
#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {

constexpr int kRsWarps = 4;
constexpr int kRsSub = 16;          // tokens per sub-tile
constexpr int kRsMaxRows = 256;     // R * G
constexpr int kRsTargetWarps = 4096;
constexpr uint32_t kNoRowRs = 0xffffffffu;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

struct RsArgs {
  const uint16_t* q;
  int R, H, G;
  const uint16_t* k_pool;
  int num_blocks, Hkv;
  const int32_t* block_table;
  int max_blocks, n_vis, n_tok;   // n_tok: tokens of pass 1 (n_vis + n_text)
  int batch, RG, MT;              // question rows per unit, 16-row tiles
  int chunk, csplit;              // tokens per CTA, CTAs per unit
  float sl2;                      // scale * log2(e)
  float* part_ml;                 // pass 1: [unit][csplit * 4][MT * 16][2]
  const float* lse2;              // pass 2: [unit][MT * 16], log2 domain
  float* scores;                  // pass 2: [unit][n_vis]
  int* status;
};

// MODE 0: per-row (max, sum) partials over tokens [0, n_tok); MODE 1: scores of
// visual tokens [0, n_vis) from lse2.
template <int D, int MODE>
__global__ void __launch_bounds__(kRsWarps * 32)
retrieve_softmax_kernel(RsArgs a) {
  grid_dep_sync();
  constexpr int KSTEPS = D / 16;
  constexpr int TILE_BYTES = kRsSub * D * 2;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* qtile = smem;                                        // [MT * 16][D] swizzled
  uint8_t* ring = smem + (size_t)a.MT * 16 * D * 2;             // [warp][2][TILE_BYTES]
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int unit = blockIdx.x / a.csplit, cta = blockIdx.x % a.csplit;
  const int b = unit / a.Hkv, g = unit % a.Hkv;
  const int n_end = MODE == 0 ? a.n_tok : a.n_vis;

  // stage the unit's question rows (row = r * G + hh), zero padding rows
  for (int i = threadIdx.x; i < a.MT * 16 * (D / 8); i += kRsWarps * 32) {
    const int row = i / (D / 8), c = i % (D / 8);
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < a.RG) {
      const int r = row / a.G, hh = row % a.G;
      v = *reinterpret_cast<const uint4*>(a.q + (((size_t)b * a.R + r) * a.H + (size_t)g * a.G + hh) * D + c * 8);
    }
    *reinterpret_cast<uint4*>(qtile + (size_t)row * D * 2 + ((c ^ (row & 7)) * 16)) = v;
  }
  __syncthreads();

  // this warp's token range: a quarter of the CTA's chunk
  const int c_begin = cta * a.chunk;
  const int c_end = min(n_end, c_begin + a.chunk);
  const int per_warp = ((a.chunk + kRsWarps - 1) / kRsWarps + kRsSub - 1) / kRsSub * kRsSub;
  const int t_begin = c_begin + wid * per_warp;
  const int t_end = min(c_end, t_begin + per_warp);
  const int nsub = t_end > t_begin ? (t_end - t_begin + kRsSub - 1) / kRsSub : 0;
  const int32_t* bt = a.block_table + (size_t)b * a.max_blocks;
  uint8_t* my = ring + (size_t)wid * 2 * TILE_BYTES;

  // row id of token t (lanes 0..15 resolve one token of a sub-tile each)
  auto resolve = [&](int t0) -> uint32_t {
    const int t = t0 + (lane & 15);
    if (t >= t_end) return kNoRowRs;
    const int page = __ldg(bt + (t >> 4));
    if (page < 0 || page >= a.num_blocks) {
      flag_status(a.status, kStatusBadBlock);
      return kNoRowRs;
    }
    return (((uint32_t)page * (uint32_t)a.Hkv + (uint32_t)g) << 4) | (uint32_t)(t & 15);
  };
  auto issue = [&](int s, uint32_t rowid) {
    const uint32_t base = smem_u32(my + (size_t)s * TILE_BYTES);
#pragma unroll
    for (int i = 0; i < kRsSub * (D / 8) / 32; ++i) {
      const int j = lane + 32 * i;
      const int tok = j / (D / 8), c = j % (D / 8);
      const uint32_t r = __shfl_sync(0xffffffffu, rowid, tok);
      const bool ok = r != kNoRowRs;
      cp_async16(base + (uint32_t)(tok * D * 2 + ((c ^ (tok & 7)) * 16)), a.k_pool + (ok ? (size_t)r * D + c * 8 : 0),
                 ok ? 16u : 0u);
    }
    cp_async_commit();
  };

  // per-row state (MODE 0): rows lane/4 and lane/4 + 8 of each query tile
  float m_r[kRsMaxRows / 16][2], l_r[kRsMaxRows / 16][2];
  if (MODE == 0) {
#pragma unroll
    for (int mt = 0; mt < kRsMaxRows / 16; ++mt) {
      m_r[mt][0] = m_r[mt][1] = -INFINITY;
      l_r[mt][0] = l_r[mt][1] = 0.f;
    }
  }
  const int mi = lane >> 3, ri = lane & 7;
  const float* lse_u = MODE == 1 ? a.lse2 + (size_t)unit * a.MT * 16 : nullptr;

  uint32_t rid_cur = 0, rid_next = 0;
  if (nsub > 0) {
    rid_cur = resolve(t_begin);
    issue(0, rid_cur);
  }
  if (nsub > 1) rid_next = resolve(t_begin + kRsSub);
  for (int it = 0; it < nsub; ++it) {
    const int s = it & 1;
    const uint32_t rid = rid_cur;
    if (it + 1 < nsub) {
      issue(s ^ 1, rid_next);
      rid_cur = rid_next;
      if (it + 2 < nsub) rid_next = resolve(t_begin + (it + 2) * kRsSub);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncwarp();
    const uint32_t kbase = smem_u32(my + (size_t)s * TILE_BYTES);
    // K fragments of the sub-tile (B operand, 16 tokens = two n-tiles)
    uint32_t bf[KSTEPS][4];
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      const int tok = (mi >> 1) * 8 + ri;
      const int c = ks * 2 + (mi & 1);
      ldsm_x4(kbase + tok * D * 2 + ((c ^ (tok & 7)) * 16), bf[ks][0], bf[ks][1], bf[ks][2], bf[ks][3]);
    }
    // token validity of the lane's four columns (n-tile nt, column tc + e)
    const int tc = (lane & 3) * 2;
    bool valid[2][2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) valid[nt][e] = __shfl_sync(0xffffffffu, rid, nt * 8 + tc + e) != kNoRowRs;

    float col[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    // query tiles unrolled so that the per-row state is indexed statically
#pragma unroll
    for (int mt = 0; mt < kRsMaxRows / 16; ++mt) {
      if (mt >= a.MT) break;
      float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        const int row = mt * 16 + (mi & 1) * 8 + ri;
        const int c = ks * 2 + (mi >> 1);
        uint32_t qa[4];
        ldsm_x4(smem_u32(qtile) + row * D * 2 + ((c ^ (row & 7)) * 16), qa[0], qa[1], qa[2], qa[3]);
        mma_16816(sacc[0], qa, bf[ks][0], bf[ks][1]);
        mma_16816(sacc[1], qa, bf[ks][2], bf[ks][3]);
      }
      if (MODE == 0) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {            // rows lane/4 (hh 0) and lane/4 + 8 (hh 1)
          float z[4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) z[nt * 2 + e] = valid[nt][e] ? sacc[nt][2 * hh + e] * a.sl2 : -INFINITY;
          float mx = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const float mn = fmaxf(m_r[mt][hh], mx);
          if (mn != -INFINITY) {
            const float ps = fast_exp2(z[0] - mn) + fast_exp2(z[1] - mn) + fast_exp2(z[2] - mn) + fast_exp2(z[3] - mn);
            l_r[mt][hh] = l_r[mt][hh] * fast_exp2(m_r[mt][hh] - mn) + ps;
            m_r[mt][hh] = mn;
          }
        }
      } else {
        const int r0 = mt * 16 + (lane >> 2);
        const float n0 = lse_u[r0], n1 = lse_u[r0 + 8];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            col[nt][e] += fast_exp2(sacc[nt][e] * a.sl2 - n0) + fast_exp2(sacc[nt][2 + e] * a.sl2 - n1);
      }
    }
    if (MODE == 1) {
      // sum over the 8 row groups (lanes with equal lane % 4), then write
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float v = col[nt][e];
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          v += __shfl_xor_sync(0xffffffffu, v, 8);
          v += __shfl_xor_sync(0xffffffffu, v, 16);
          const int t = t_begin + it * kRsSub + nt * 8 + tc + e;
          if (lane < 4 && valid[nt][e] && t < t_end) a.scores[(size_t)unit * a.n_vis + t] = v;
        }
    }
    __syncwarp();
  }

  if (MODE == 0) {
    // per-row partials of this warp's range (rows lane/4, +8; quad lanes share a row)
    const int split = cta * kRsWarps + wid;
    const int nsplit = a.csplit * kRsWarps;
#pragma unroll
    for (int mm = 0; mm < kRsMaxRows / 16; ++mm) {
      if (mm >= a.MT) break;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float l = l_r[mm][hh];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        if ((lane & 3) == 0) {
          const int row = mm * 16 + (lane >> 2) + 8 * hh;
          float* p = a.part_ml + (((size_t)unit * nsplit + split) * a.MT * 16 + row) * 2;
          p[0] = m_r[mm][hh];
          p[1] = l;
        }
      }
    }
  }
}

// lse2[unit][row] from the pass-1 partials (merged in split order), or from a
// caller's natural-log lse [B][R][H]; padding rows get +inf (no mass).
__global__ void retrieve_softmax_lse_kernel(const float* __restrict__ part_ml, int nsplit, const float* __restrict__ lse_in,
                                            int R, int H, int G, int Hkv, int RG, int MT, float* __restrict__ lse2) {
  grid_dep_sync();
  const int unit = blockIdx.x;
  const int b = unit / Hkv, g = unit % Hkv;
  for (int row = threadIdx.x; row < MT * 16; row += blockDim.x) {
    float out = INFINITY;
    if (row < RG) {
      if (lse_in) {
        const int r = row / G, hh = row % G;
        out = lse_in[((size_t)b * R + r) * H + (size_t)g * G + hh] * kLog2e;
      } else {
        float M = -INFINITY;
        for (int s = 0; s < nsplit; ++s)
          M = fmaxf(M, part_ml[(((size_t)unit * nsplit + s) * MT * 16 + row) * 2]);
        float L = 0.f;
        for (int s = 0; s < nsplit; ++s) {
          const float* p = part_ml + (((size_t)unit * nsplit + s) * MT * 16 + row) * 2;
          if (p[0] != -INFINITY) L += p[1] * fast_exp2(p[0] - M);
        }
        out = L > 0.f ? M + __log2f(L) : INFINITY;
      }
    }
    lse2[(size_t)unit * MT * 16 + row] = out;
  }
}

struct RsPlan {
  int chunk, csplit;
};

RsPlan rs_plan(int units, int n) {
  // about kRsTargetWarps warps over the GPU, at least 64 tokens per warp
  long long warps = (long long)units * ((n + 63) / 64);
  RsPlan p;
  long long per_warp = 64;
  if (warps > kRsTargetWarps) per_warp = ((long long)units * n + kRsTargetWarps - 1) / kRsTargetWarps;
  per_warp = (per_warp + kRsSub - 1) / kRsSub * kRsSub;
  p.chunk = (int)(per_warp * kRsWarps);
  p.csplit = n > 0 ? (n + p.chunk - 1) / p.chunk : 1;
  return p;
}

size_t rs_smem(int D, int MT) { return (size_t)MT * 16 * D * 2 + (size_t)kRsWarps * 2 * kRsSub * D * 2; }

}  // namespace

size_t retrieve_softmax_workspace_bytes(int B, int R, int H, int Hkv, int D, int n_vis, int n_text) {
  const long long units = (long long)B * Hkv;
  const int G = Hkv > 0 ? H / Hkv : 1;
  const int MT = (R * G + 15) / 16;
  const RsPlan p1 = rs_plan((int)units, n_vis + n_text);
  const size_t parts = (size_t)units * p1.csplit * kRsWarps * MT * 16 * 2 * sizeof(float);
  const size_t lse = (size_t)units * MT * 16 * sizeof(float);
  const size_t sc = (size_t)units * n_vis * sizeof(float);
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  (void)D;
  return r256(parts) + r256(lse) + r256(sc);
}

int retrieve_softmax_max_rows() { return kRsMaxRows; }

cudaError_t launch_retrieve_softmax(const void* q, int R, int H, float scale, const void* k_pool, int num_blocks,
                                    int Hkv, int D, const int32_t* block_table, int max_blocks, int n_vis,
                                    int n_text, int batch, const float* lse_in, int k, int32_t* vis_idx,
                                    float* scores_out, void* ws, int* status, cudaStream_t stream) {
  const int units = batch * Hkv;
  if (units == 0) return cudaSuccess;
  const int G = H / Hkv, RG = R * G, MT = (RG + 15) / 16;
  const RsPlan p1 = rs_plan(units, n_vis + n_text);
  auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* w = static_cast<uint8_t*>(ws);
  float* part_ml = reinterpret_cast<float*>(w);
  float* lse2 = reinterpret_cast<float*>(w + r256((size_t)units * p1.csplit * kRsWarps * MT * 16 * 2 * sizeof(float)));
  float* sc_ws = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(lse2) + r256((size_t)units * MT * 16 * sizeof(float)));
  float* scores = scores_out ? scores_out : sc_ws;

  RsArgs a;
  a.q = static_cast<const uint16_t*>(q);
  a.R = R; a.H = H; a.G = G;
  a.k_pool = static_cast<const uint16_t*>(k_pool);
  a.num_blocks = num_blocks; a.Hkv = Hkv;
  a.block_table = block_table; a.max_blocks = max_blocks;
  a.n_vis = n_vis; a.n_tok = n_vis + n_text;
  a.batch = batch; a.RG = RG; a.MT = MT;
  a.sl2 = scale * kLog2e;
  a.part_ml = part_ml; a.lse2 = lse2; a.scores = scores; a.status = status;
  const size_t smem = rs_smem(D, MT);
  cudaError_t e;
  auto set_smem = [&](const void* fn) {
    return smem > 48 * 1024 ? cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
                            : cudaSuccess;
  };
  if (!lse_in) {
    a.chunk = p1.chunk; a.csplit = p1.csplit;
    if (D == 128) {
      if ((e = set_smem((const void*)retrieve_softmax_kernel<128, 0>)) != cudaSuccess) return e;
      e = launch_dependent(retrieve_softmax_kernel<128, 0>, dim3(units * p1.csplit), dim3(kRsWarps * 32), smem, stream, a);
    } else {
      if ((e = set_smem((const void*)retrieve_softmax_kernel<64, 0>)) != cudaSuccess) return e;
      e = launch_dependent(retrieve_softmax_kernel<64, 0>, dim3(units * p1.csplit), dim3(kRsWarps * 32), smem, stream, a);
    }
    if (e != cudaSuccess) return e;
  }
  e = launch_dependent(retrieve_softmax_lse_kernel, dim3(units), dim3(256), 0, stream, part_ml, p1.csplit * kRsWarps,
                       lse_in, R, H, G, Hkv, RG, MT, lse2);
  if (e != cudaSuccess) return e;
  const RsPlan p2 = rs_plan(units, n_vis);
  a.chunk = p2.chunk; a.csplit = p2.csplit;
  if (D == 128) {
    if ((e = set_smem((const void*)retrieve_softmax_kernel<128, 1>)) != cudaSuccess) return e;
    e = launch_dependent(retrieve_softmax_kernel<128, 1>, dim3(units * p2.csplit), dim3(kRsWarps * 32), smem, stream, a);
  } else {
    if ((e = set_smem((const void*)retrieve_softmax_kernel<64, 1>)) != cudaSuccess) return e;
    e = launch_dependent(retrieve_softmax_kernel<64, 1>, dim3(units * p2.csplit), dim3(kRsWarps * 32), smem, stream, a);
  }
  if (e != cudaSuccess) return e;
  if (topk_prefers_cluster(n_vis)) return launch_topk_cluster(scores, units, n_vis, k, vis_idx, stream);
  return launch_topk_rows(scores, units, n_vis, k, vis_idx, stream);
}

}  // namespace sv
