// Query-agnostic prefill salience on the tcgen05 tensor cores.
//
// velog.io SparseVILA summary §3.1: for encoders without a summary token
// (SigLIP, QwenVL) a token's salience is the intra-visual attention it
// receives, averaged over all tokens; the kernel paragraph streams the softmax
// normalisation and the salience accumulation without materialising the
// N x N attention matrix.  xllm-io review §三 gives the formula.  Per frame b:
//   s[b][j] = 1/(H N) sum_h sum_i exp(scale q_i.k_j - lse_i),
//   lse_i   = log sum_j exp(scale q_i.k_j).
//
// Design (one CTA per (frame, head), 16 softmax warps + 1 TMA/MMA warp):
//   pass 1  K_h resident in shared memory, 128-row tiles of Q_h streamed by
//           TMA; S = Q_tile K^T (M=128, N<=256 per MMA, K=d padded to 16) goes
//           to a double-buffered TMEM accumulator; every softmax thread owns
//           one query row (one TMEM lane) and a quarter of the columns, keeps
//           an online max / sum of exp2, and the four parts are merged into
//           lse_i (log2 domain) in shared memory.
//   The element-wise work is exp-bound: it uses packed fp32x2 FMA/ADD, a
//   3-input max tree, independent accumulators, and sends a fixed fraction
//   of the exponentials to an FMA-pipe polynomial (fastmath.cuh) so that
//   MUFU and the FMA pipe share the load.
//   pass 2  Q_h resident, 128-row tiles of K_h streamed; S^T = K_tile Q^T puts
//           one key per TMEM lane, so the column sum over queries becomes a
//           per-thread row sum of exp2(z - lse_i) with lse_i broadcast from
//           shared memory.  Padded queries carry lse = +inf and contribute 0.
// Shared-memory operands use the K-major no-swizzle layout (8x16-byte core
// matrices); TMA writes them directly with 8-element x 128-row boxes, and out
// of range rows are zero-filled by TMA.  Head dims that are not a multiple of
// 16 (72) get a zero K-chunk that TMA never writes.
// Per-head column sums go to the workspace; a second kernel averages heads in
// a fixed order (deterministic).
#include "common.cuh"
#include "kernels.h"
#include "fastmath.cuh"
#include "tc_ptx.cuh"

namespace sv {

namespace {

#ifndef SV_SAL_SOFT_WARPS
#define SV_SAL_SOFT_WARPS 16
#endif
constexpr int kSoftWarps = SV_SAL_SOFT_WARPS;
constexpr int kParts = kSoftWarps / 4;   // column parts per TMEM lane quarter
constexpr int kPartCols = 256 / kParts;  // columns of a 256-column chunk per warp
#ifndef SV_SAL_POLY_PAIRS
#define SV_SAL_POLY_PAIRS 0
#endif
// of every 16 element pairs, this many take exp2 on the FMA pipe, the rest on MUFU
constexpr int kPolyPairs = SV_SAL_POLY_PAIRS;
constexpr int kThreads = (kSoftWarps + 1) * 32;
constexpr int kTileRows = 128;
constexpr int kChunkCols = 256;
constexpr int kTmemCols = 512;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kStatusSalTimeout = 0x10;

struct SalGeom {
  int Kp;       // padded head dim (multiple of 16)
  int kc_load;  // 8-element K chunks that TMA loads (d / 8)
  int Np;       // N rounded up to 32 (columns that MMAs produce)
  int Rr;       // N rounded up to 128 (rows of a resident operand)
  int nt;       // 128-row tiles
  int nchunks;  // 256-column chunks
  size_t res_bytes, slot_bytes, smem_bytes;
};

SalGeom sal_geom(int N, int d) {
  SalGeom g;
  g.Kp = (d + 15) / 16 * 16;
  g.kc_load = d / 8;
  g.Np = (N + 31) / 32 * 32;
  g.Rr = (N + kTileRows - 1) / kTileRows * kTileRows;
  g.nt = g.Rr / kTileRows;
  g.nchunks = (g.Np + kChunkCols - 1) / kChunkCols;
  g.res_bytes = (size_t)g.Rr * g.Kp * 2;
  g.slot_bytes = (size_t)kTileRows * g.Kp * 2;
  g.smem_bytes = 1024 + g.res_bytes + 2 * g.slot_bytes + (size_t)g.Rr * 4 + 2 * kParts * 256 * 4;
  return g;
}

// Every CTA allocates all 512 TMEM columns, so the launch asks for more than
// half of an SM's shared memory: one CTA per SM, no CTA ever waits in alloc.
size_t launch_smem(const SalGeom& g) {
  const size_t one_per_sm = 120 * 1024;
  return g.smem_bytes > one_per_sm ? g.smem_bytes : one_per_sm;
}

struct SalArgs {
  int N, Kp, kc_load, ks_steps, Np, Rr, nt, nchunks;
  float sl2;  // scale * log2(e)
  float* colsum;
  int* status;
};

struct SalShared {
  uint64_t bar_res, bar_pass, bar_done;
  uint64_t bar_slot[2], bar_free[2], bar_full[2], bar_empty[2];
  uint32_t tmem_base;
  int abort_flag;
};

// Bounded wait: returns immediately once the CTA has aborted.  The timer is
// read only when the phase is not already complete (reading it is slow).
__device__ __forceinline__ void wait_bar(uint64_t* bar, uint32_t parity, SalShared& sh) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::global_timer();
  for (uint32_t it = 0;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return;
    if ((it & 127) == 127) {
      if (*(volatile int*)&sh.abort_flag) return;
      if (ptx::global_timer() - t0 > kWaitLimitNs) {
        *(volatile int*)&sh.abort_flag = 1;
        return;
      }
    }
  }
}

__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kSoftWarps * 32) : "memory"); }

__global__ void __launch_bounds__(kThreads, 1)
salience_colsum_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       SalArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ SalShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int Kp = a.Kp, Rr = a.Rr;
  uint8_t* res = smem;
  uint8_t* slot[2] = {smem + (size_t)Rr * Kp * 2, smem + (size_t)Rr * Kp * 2 + kTileRows * Kp * 2};
  float* nlse2 = reinterpret_cast<float*>(slot[1] + kTileRows * Kp * 2);
  float* mrg = nlse2 + Rr;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int unit = blockIdx.x;

  // zero the K chunks that TMA never writes (head dim padded to 16)
  for (int kc = a.kc_load; kc < Kp / 8; ++kc) {
    uint4* r = reinterpret_cast<uint4*>(res + (size_t)kc * Rr * 16);
    for (int i = threadIdx.x; i < Rr; i += blockDim.x) r[i] = make_uint4(0, 0, 0, 0);
    for (int s = 0; s < 2; ++s) {
      uint4* p = reinterpret_cast<uint4*>(slot[s] + (size_t)kc * kTileRows * 16);
      for (int i = threadIdx.x; i < kTileRows; i += blockDim.x) p[i] = make_uint4(0, 0, 0, 0);
    }
  }
  ptx::fence_proxy_async_smem();

  if (threadIdx.x == 0) {
    ptx::mbar_init(&sh.bar_res, 1);
    ptx::mbar_init(&sh.bar_pass, 1);
    ptx::mbar_init(&sh.bar_done, 1);
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&sh.bar_slot[i], 1);
      ptx::mbar_init(&sh.bar_free[i], 1);
      ptx::mbar_init(&sh.bar_full[i], 1);
      ptx::mbar_init(&sh.bar_empty[i], kSoftWarps);
    }
    sh.abort_flag = 0;
    ptx::mbar_fence_init();
  }
  if (warp == 0) ptx::tmem_alloc(&sh.tmem_base, kTmemCols);
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = sh.tmem_base;

  if (warp == kSoftWarps) {
    // ------------------------------------------------ TMA + MMA issue (one thread)
    if (lane == 0) {
      ptx::prefetch_tensormap(&tq);
      ptx::prefetch_tensormap(&tk);
      const uint32_t tile_tx = (uint32_t)a.kc_load * kTileRows * 16;
      auto load_rows = [&](const CUtensorMap* map, uint8_t* dst, int dst_rows, int row0, int nrows,
                           uint64_t* bar) {
        ptx::mbar_arrive_expect_tx(bar, tile_tx * (uint32_t)(nrows / kTileRows));
        for (int r = 0; r < nrows; r += kTileRows)
          for (int kc = 0; kc < a.kc_load; ++kc)
            ptx::tma_load_3d(dst + (size_t)kc * dst_rows * 16 + (size_t)r * 16, map, kc * 8,
                             row0 + r, unit, bar);
      };
      uint32_t u = 0;                      // TMEM buffer uses
      uint32_t slot_waits[2] = {0, 0}, free_waits[2] = {0, 0};
      const uint32_t res_base = ptx::smem_addr(res);
      for (int pass = 0; pass < 2; ++pass) {
        const CUtensorMap* res_map = pass == 0 ? &tk : &tq;
        const CUtensorMap* str_map = pass == 0 ? &tq : &tk;
        if (pass == 1) {  // resident operand and slots are rewritten: drain pass-1 MMAs
          ptx::mma_commit(&sh.bar_pass);
          wait_bar(&sh.bar_pass, 0, sh);
        }
        load_rows(res_map, res, Rr, 0, Rr, &sh.bar_res);
        load_rows(str_map, slot[0], kTileRows, 0, kTileRows, &sh.bar_slot[0]);
        if (a.nt > 1) load_rows(str_map, slot[1], kTileRows, kTileRows, kTileRows, &sh.bar_slot[1]);
        wait_bar(&sh.bar_res, (uint32_t)pass, sh);
        for (int t = 0; t < a.nt; ++t) {
          const int s = t & 1;
          wait_bar(&sh.bar_slot[s], slot_waits[s]++ & 1, sh);
          const uint32_t a_base = ptx::smem_addr(slot[s]);
          for (int c = 0; c < a.nchunks; ++c, ++u) {
            const uint32_t buf = u & 1;
            if (u >= 2) wait_bar(&sh.bar_empty[buf], ((u >> 1) - 1) & 1, sh);
            ptx::tc_fence_after();
            const int nc = min(kChunkCols, a.Np - kChunkCols * c);
            const uint32_t idesc = ptx::idesc_bf16_f32(kTileRows, nc);
            for (int ks = 0; ks < a.ks_steps; ++ks) {
              const uint64_t ad = ptx::smem_desc_kmajor(a_base + 2 * ks * kTileRows * 16,
                                                        kTileRows * 16, 128);
              const uint64_t bd = ptx::smem_desc_kmajor(
                  res_base + 2 * ks * Rr * 16 + kChunkCols * c * 16, (uint32_t)Rr * 16, 128);
              ptx::mma_bf16(tbase + buf * kChunkCols, ad, bd, idesc, ks > 0 ? 1u : 0u);
            }
            ptx::mma_commit(&sh.bar_full[buf]);
          }
          if (t + 2 < a.nt) {
            ptx::mma_commit(&sh.bar_free[s]);
            wait_bar(&sh.bar_free[s], free_waits[s]++ & 1, sh);
            load_rows(str_map, slot[s], kTileRows, (t + 2) * kTileRows, kTileRows,
                      &sh.bar_slot[s]);
          }
        }
      }
      ptx::mma_commit(&sh.bar_done);
      wait_bar(&sh.bar_done, 0, sh);
    }
  } else {
    // ------------------------------------------------ softmax warps
    // warp w reads TMEM lane quarter (w & 3) -- the hardware ties a warp to the
    // lanes 32 * (w % 4) .. + 31 -- and the column part (w >> 2) of a chunk.
    const int quarter = warp & 3, part = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const float sl2 = a.sl2;
    const uint64_t sl2x2 = fm::splat2(sl2);
    uint32_t u = 0;
    uint32_t ra[32], rb[32];
    // Runs fn(group registers, column offset) on the warp's ng 32-column
    // groups starting at TMEM address ta, with the next group's TMEM load in
    // flight while the current one is processed.
    auto for_groups = [&](uint32_t ta, int ng, auto&& fn) {
      if (ng <= 0) return;
      ptx::tmem_ld32(ta, ra);
      ptx::tmem_wait_ld(ra);
      if (ng > 1) ptx::tmem_ld32(ta + 32, rb);
      fn(ra, 0);
      if (ng > 1) {
        ptx::tmem_wait_ld(rb);
        if (ng > 2) ptx::tmem_ld32(ta + 64, ra);
        fn(rb, 32);
      }
      if (ng > 2) {
        ptx::tmem_wait_ld(ra);
        if (ng > 3) ptx::tmem_ld32(ta + 96, rb);
        fn(ra, 64);
      }
      if (ng > 3) {
        ptx::tmem_wait_ld(rb);
        fn(rb, 96);
      }
    };
    // pass 1: row log-sum-exp (log2 domain)
    for (int t = 0; t < a.nt; ++t) {
      const bool live = t * kTileRows + quarter * 32 < a.N;
      float m = -INFINITY, l = 0.f;
      for (int c = 0; c < a.nchunks; ++c, ++u) {
        const uint32_t buf = u & 1;
        wait_bar(&sh.bar_full[buf], (u >> 1) & 1, sh);
        ptx::tc_fence_after();
        const int nc = min(kChunkCols, a.Np - kChunkCols * c);
        const int col0 = part * kPartCols;
        const int ncols = live ? max(0, min(kPartCols, nc - col0)) : 0;
        {
          const uint32_t ta = tbase + lane_addr + buf * kChunkCols + col0;
          for_groups(ta, ncols >> 5, [&](uint32_t* v, int g) {
            const int key0 = kChunkCols * c + col0 + g;
            if (key0 + 32 > a.N) {
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (key0 + i >= a.N) v[i] = __float_as_uint(-INFINITY);
            }
            float mx[11];
#pragma unroll
            for (int i = 0; i < 10; ++i)
              mx[i] = fm::max3(__uint_as_float(v[3 * i]), __uint_as_float(v[3 * i + 1]),
                               __uint_as_float(v[3 * i + 2]));
            mx[10] = fmaxf(__uint_as_float(v[30]), __uint_as_float(v[31]));
            const float cm = fmaxf(fm::max3(fm::max3(mx[0], mx[1], mx[2]), fm::max3(mx[3], mx[4], mx[5]),
                                            fm::max3(mx[6], mx[7], mx[8])),
                                   fmaxf(mx[9], mx[10]));
            // stale running max: rescale only when the group max exceeds it by
            // more than 8 (log2 units), so the exps need not wait for the max
            const float cms = cm * sl2;
            if (cms > m + 8.0f) {
              l = l * fm::ex2_mufu(m - cms);
              m = cms;
            }
            if (m == -INFINITY) return;
            const uint64_t nmn = fm::splat2(-m);
            uint64_t acc[4] = {0, 0, 0, 0};
#pragma unroll
            for (int pr = 0; pr < 16; ++pr) {
              const uint64_t x = fm::fma2(fm::pack2(__uint_as_float(v[2 * pr]), __uint_as_float(v[2 * pr + 1])),
                                          sl2x2, nmn);
              const uint64_t e = pr < kPolyPairs ? fm::exp2_poly2(x) : fm::exp2_mufu2(x);
              acc[pr & 3] = fm::add2(acc[pr & 3], e);
            }
            const uint64_t s2 = fm::add2(fm::add2(acc[0], acc[1]), fm::add2(acc[2], acc[3]));
            float s0, s1;
            fm::unpack2(s2, s0, s1);
            l += s0 + s1;
          });
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sh.bar_empty[buf]);
      }
      float* mg = mrg + (t & 1) * (kParts * 256);
      mg[part * 256 + row * 2] = m;
      mg[part * 256 + row * 2 + 1] = l;
      softmax_bar();
      if (part == 0) {
        float M = -INFINITY;
#pragma unroll
        for (int p2 = 0; p2 < kParts; ++p2) M = fmaxf(M, mg[p2 * 256 + row * 2]);
        float L = 0.f;
#pragma unroll
        for (int p2 = 0; p2 < kParts; ++p2) {
          const float mp = mg[p2 * 256 + row * 2];
          if (mp != -INFINITY) L += mg[p2 * 256 + row * 2 + 1] * fm::ex2_mufu(mp - M);
        }
        const int qi = t * kTileRows + row;
        // stored negated: pass 2 adds it with one packed FMA; padded queries
        // get -inf and contribute nothing
        nlse2[qi] = qi < a.N ? -(M + __log2f(L)) : -INFINITY;
      }
    }
    softmax_bar();
    // pass 2: column sums of exp2(z - lse), one key per TMEM lane
    for (int t = 0; t < a.nt; ++t) {
      const bool live = t * kTileRows + quarter * 32 < a.N;
      uint64_t acc[4] = {0, 0, 0, 0};
      for (int c = 0; c < a.nchunks; ++c, ++u) {
        const uint32_t buf = u & 1;
        wait_bar(&sh.bar_full[buf], (u >> 1) & 1, sh);
        ptx::tc_fence_after();
        const int nc = min(kChunkCols, a.Np - kChunkCols * c);
        const int col0 = part * kPartCols;
        const int ncols = live ? max(0, min(kPartCols, nc - col0)) : 0;
        {
          const uint32_t ta = tbase + lane_addr + buf * kChunkCols + col0;
          for_groups(ta, ncols >> 5, [&](const uint32_t* v, int g) {
            const uint64_t* nl = reinterpret_cast<const uint64_t*>(nlse2 + kChunkCols * c + col0 + g);
#pragma unroll
            for (int pr = 0; pr < 16; ++pr) {
              const uint64_t x = fm::fma2(fm::pack2(__uint_as_float(v[2 * pr]), __uint_as_float(v[2 * pr + 1])),
                                          sl2x2, nl[pr]);
              const uint64_t e = pr < kPolyPairs ? fm::exp2_poly2(x) : fm::exp2_mufu2(x);
              acc[pr & 3] = fm::add2(acc[pr & 3], e);
            }
          });
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sh.bar_empty[buf]);
      }
      const uint64_t s2 = fm::add2(fm::add2(acc[0], acc[1]), fm::add2(acc[2], acc[3]));
      float s0, s1;
      fm::unpack2(s2, s0, s1);
      float* mg = mrg + (t & 1) * (kParts * 128);
      mg[part * 128 + row] = s0 + s1;
      softmax_bar();
      if (part == 0) {
        const int key = t * kTileRows + row;
        float tot = 0.f;
#pragma unroll
        for (int p2 = 0; p2 < kParts; ++p2) tot += mg[p2 * 128 + row];
        if (key < a.N) a.colsum[(size_t)unit * a.N + key] = tot;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sh.abort_flag) flag_status(a.status, kStatusSalTimeout);
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tbase, kTmemCols);
  }
}

// s[b][j] = (1 / (H N)) * sum_h colsum[b][h][j], heads summed in order.
__global__ void salience_head_mean_kernel(const float* __restrict__ colsum, int B, int H, int N,
                                          float inv, float* __restrict__ out) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)B * N) return;
  const long long b = i / N, j = i % N;
  const float* p = colsum + b * H * (long long)N + j;
  float s = 0.f;
  for (int h = 0; h < H; ++h) s += p[(long long)h * N];
  out[i] = s * inv;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool make_map(CUtensorMap* map, const void* base, int d, int N, int units) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)units};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
  cuuint32_t box[3] = {8, (cuuint32_t)kTileRows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t salience_smem_bytes(int N, int d) { return launch_smem(sal_geom(N, d)); }

size_t salience_workspace_bytes(int B, int H, int N, int d) {
  (void)d;
  return (size_t)B * H * N * sizeof(float);
}

cudaError_t launch_salience(const void* q, const void* k, int B, int H, int N, int d, float scale,
                            float* salience, void* ws, int* status, int num_sms,
                            cudaStream_t stream) {
  (void)num_sms;
  const SalGeom g = sal_geom(N, d);
  CUtensorMap tq, tk;
  if (!make_map(&tq, q, d, N, B * H) || !make_map(&tk, k, d, N, B * H)) return cudaErrorInvalidValue;
  SalArgs a;
  a.N = N;
  a.Kp = g.Kp;
  a.kc_load = g.kc_load;
  a.ks_steps = g.Kp / 16;
  a.Np = g.Np;
  a.Rr = g.Rr;
  a.nt = g.nt;
  a.nchunks = g.nchunks;
  a.sl2 = scale * kLog2e;
  a.colsum = static_cast<float*>(ws);
  a.status = status;
  const size_t smem = launch_smem(g);
  cudaError_t e = cudaFuncSetAttribute(salience_colsum_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  salience_colsum_kernel<<<B * H, kThreads, smem, stream>>>(tq, tk, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long total = (long long)B * N;
  salience_head_mean_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(
      a.colsum, B, H, N, 1.0f / ((float)H * (float)N), salience);
  return cudaGetLastError();
}

}  // namespace sv
