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
// Design: persistent CTAs (one per SM), each walking over (frame, head)
// units; 16 softmax warps, one MMA-issue warp and one TMA warp.  Per unit two
// passes run back to back over 128-row tiles x 256-column chunks:
//   pass 1  K_h resident in shared memory, 128-row tiles of Q_h streamed by
//           TMA; S = Q_tile K_chunk^T (M=128, N<=256, K=d padded to 16) goes
//           to one of two 256-column TMEM buffers; every softmax thread owns
//           one query row (one TMEM lane) of a 64-column slice of the chunk
//           and keeps an online max / sum of exp2 (log2 domain); per tile the
//           four slice log-sum-exps of a row are merged into lse_i in shared
//           memory.
//   pass 2  Q_h resident, 128-row tiles of K_h streamed; S^T = K_tile Q^T puts
//           one key per TMEM lane, so the column sum over queries becomes a
//           per-thread row sum of exp2(z - lse_i) with lse_i broadcast from
//           shared memory.  Padded queries carry lse = +inf and contribute 0.
// Chunk u of the whole sequence goes to TMEM buffer u % 2; all 16 softmax
// warps read every chunk (warp w: lane quarter w % 4, slice w / 4), so while
// they work through one buffer the MMAs refill the other, and no warp waits
// for the refill of "its" buffer.  One N=256 MMA costs about as much as one
// N=128 MMA here, so the 256-column chunks halve the tensor-pipe time.
// The resident operand is replaced chunk by chunk: as soon as the last tile's
// MMAs on a 128-row chunk complete, the TMA warp loads the next pass's (or the
// next unit's) rows there, so the tensor pipe never drains between passes.
// The MMA warp runs its schedule with the whole warp (uniform control flow)
// and issues from one elected lane; waiting warps sleep inside try_wait.
// The element-wise work is bound by exp throughput and instruction issue: it
// uses packed fp32x2 FMA/ADD, a 3-input max tree, a stale running max
// (rescaled only when it grows by more than 8), one 32-column group in
// registers at a time and one accumulator chain; variants with
// double-buffered TMEM loads, more accumulator chains, scalar arithmetic,
// 24 softmax warps or buffers tied to warps measured slower on the SigLIP
// shape.
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

// Work split (chosen by measurement on the SigLIP shape; see the notes at the
// top): two 256-column TMEM buffers filled by N=256 MMAs; every softmax warp
// reads a fixed 64-column slice of every chunk, 32-column groups loaded one
// at a time and summed into one fp32x2 accumulator.
constexpr int kBufs = 2;                       // TMEM buffers (one chunk each)
constexpr int kBufCols = 256;                  // columns of one TMEM buffer (N of one MMA)
constexpr int kPieces = kBufCols / 128;        // 128-row resident pieces per chunk
constexpr int kSlices = 4;                     // softmax warps per TMEM lane quarter
constexpr int kWarpCols = kBufCols / kSlices;  // columns of every chunk per softmax warp
static_assert(kWarpCols % 32 == 0, "slices are whole 32-column groups");
constexpr int kParts = kSlices;                // row partials per lane (one per slice)
constexpr int kSoftWarps = 4 * kSlices;
constexpr int kSlots = 2;        // streamed 128-row operand tiles in flight
constexpr int kMmaWarp = kSoftWarps, kTmaWarp = kSoftWarps + 1;
constexpr int kThreads = (kSoftWarps + 2) * 32;
constexpr int kTileRows = 128;
constexpr int kTmemCols = 512;  // allocations are powers of two; kBufs * kBufCols <= 512
static_assert(kBufs * kBufCols <= kTmemCols, "TMEM buffers exceed the allocation");
static_assert(kThreads <= 1024, "block too large");
constexpr int kMaxChunks = 64;   // resident chunks (N <= 8192; shared memory caps N far lower)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

struct SalGeom {
  int Kp;       // padded head dim (multiple of 16)
  int kc_load;  // 8-element K chunks that TMA loads (d / 8)
  int Np;       // N rounded up to 32 (columns that MMAs produce)
  int Rr;       // N rounded up to 128 (rows of a resident operand)
  int nt;       // 128-row tiles = 128-row resident pieces
  size_t res_bytes, slot_bytes, smem_bytes;
};

SalGeom sal_geom(int N, int d) {
  SalGeom g;
  g.Kp = (d + 15) / 16 * 16;
  g.kc_load = d / 8;
  g.Np = (N + 31) / 32 * 32;
  g.Rr = (N + kTileRows - 1) / kTileRows * kTileRows;
  g.nt = g.Rr / kTileRows;
  g.res_bytes = (size_t)g.Rr * g.Kp * 2;
  g.slot_bytes = (size_t)kTileRows * g.Kp * 2;
  // operands, per-part row partials, per-row lse
  g.smem_bytes = 1024 + g.res_bytes + kSlots * g.slot_bytes + (size_t)kParts * g.Rr * 4 + (size_t)g.Rr * 4;
  return g;
}

// Every CTA allocates all 512 TMEM columns, so the launch asks for more than
// half of an SM's shared memory: one CTA per SM, no CTA ever waits in alloc.
size_t launch_smem(const SalGeom& g) {
  const size_t one_per_sm = 120 * 1024;
  return g.smem_bytes > one_per_sm ? g.smem_bytes : one_per_sm;
}

struct SalArgs {
  int N, Kp, kc_load, ks_steps, Np, Rr, nt, units;
  float sl2;  // scale * log2(e)
  float* colsum;
  int* status;
};

struct SalShared {
  uint64_t bar_done;
  uint64_t bar_slot[kSlots], bar_slot_free[kSlots];
  uint64_t bar_full[kBufs], bar_empty[kBufs];
  uint64_t bar_res[kMaxChunks], bar_res_free[kMaxChunks];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr uint32_t kSuspendHintNs = 100000;  // try_wait sleep limit per poll
// Bounded wait: returns immediately once the CTA has aborted.  A waiting warp
// sleeps inside try_wait (woken when the phase completes) instead of spinning
// on issue slots that working warps of the same SM sub-partition need.
__device__ __forceinline__ void wait_bar(uint64_t* bar, uint32_t parity, SalShared& sh) {
  if (ptx::mbar_try_wait(bar, parity)) return;
  const uint64_t t0 = ptx::global_timer();
  for (;;) {
    if (ptx::mbar_try_wait_sleep(bar, parity, kSuspendHintNs)) return;
    if (*(volatile int*)&sh.abort_flag) return;
    if (ptx::global_timer() - t0 > kWaitLimitNs) {
      *(volatile int*)&sh.abort_flag = 1;
      return;
    }
  }
}

// One 128 x nc chunk: KS K-steps of 16, descriptors stepped in their low halves.
template <int KS>
__device__ __forceinline__ void mma_chunk(uint32_t d_t, uint32_t a_lo, uint32_t b_lo, uint32_t hi,
                                          uint32_t a_ks, uint32_t b_ks, uint32_t idesc) {
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
    ptx::mma_bf16_split(d_t, a_lo + ks * a_ks, b_lo + ks * b_ks, hi, idesc, ks > 0 ? 1u : 0u);
}

__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kSoftWarps * 32) : "memory"); }

__global__ void __launch_bounds__(kThreads, 1)
salience_colsum_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       SalArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ SalShared sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int Kp = a.Kp, Rr = a.Rr, nt = a.nt;
  uint8_t* res = smem;
  uint8_t* slots = smem + (size_t)Rr * Kp * 2;
  const size_t slot_bytes = (size_t)kTileRows * Kp * 2;
  float* part_lse = reinterpret_cast<float*>(slots + kSlots * slot_bytes);  // [kParts][Rr]
  float* nlse2 = part_lse + kParts * Rr;                                     // [Rr]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // zero the K chunks that TMA never writes (head dim padded to 16)
  for (int kc = a.kc_load; kc < Kp / 8; ++kc) {
    uint4* r = reinterpret_cast<uint4*>(res + (size_t)kc * Rr * 16);
    for (int i = threadIdx.x; i < Rr; i += blockDim.x) r[i] = make_uint4(0, 0, 0, 0);
    for (int s = 0; s < kSlots; ++s) {
      uint4* p = reinterpret_cast<uint4*>(slots + s * slot_bytes + (size_t)kc * kTileRows * 16);
      for (int i = threadIdx.x; i < kTileRows; i += blockDim.x) p[i] = make_uint4(0, 0, 0, 0);
    }
  }
  ptx::fence_proxy_async_smem();

  if (threadIdx.x == 0) {
    ptx::mbar_init(&sh.bar_done, 1);
    for (int i = 0; i < kSlots; ++i) {
      ptx::mbar_init(&sh.bar_slot[i], 1);
      ptx::mbar_init(&sh.bar_slot_free[i], 1);
    }
    for (int i = 0; i < kBufs; ++i) {
      ptx::mbar_init(&sh.bar_full[i], 1);
      ptx::mbar_init(&sh.bar_empty[i], kSoftWarps);  // every softmax warp reads every chunk
    }
    for (int i = 0; i < nt; ++i) {
      ptx::mbar_init(&sh.bar_res[i], 1);
      ptx::mbar_init(&sh.bar_res_free[i], 1);
    }
    sh.abort_flag = 0;
    ptx::mbar_fence_init();
  }
  if (warp == 0) ptx::tmem_alloc(&sh.tmem_base, kTmemCols);
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = sh.tmem_base;

  if (warp == kTmaWarp) {
    // ------------------------------------------------ TMA loads (one thread)
    if (lane == 0) {
      ptx::prefetch_tensormap(&tq);
      ptx::prefetch_tensormap(&tk);
      const uint32_t tile_tx = (uint32_t)a.kc_load * kTileRows * 16;
      auto load_rows = [&](const CUtensorMap* map, uint8_t* dst, int dst_rows, int row0, int unit,
                           uint64_t* bar) {
        ptx::mbar_arrive_expect_tx(bar, tile_tx);
        for (int kc = 0; kc < a.kc_load; ++kc)
          ptx::tma_load_3d(dst + (size_t)kc * dst_rows * 16, map, kc * 8, row0, unit, bar);
      };
      uint32_t g = 0, phase = 0;  // streamed tiles, passes issued so far
      for (int unit = blockIdx.x; unit < a.units; unit += gridDim.x) {
        for (int pass = 0; pass < 2; ++pass, ++phase) {
          const CUtensorMap* res_map = pass == 0 ? &tk : &tq;
          const CUtensorMap* str_map = pass == 0 ? &tq : &tk;
          auto load_tile = [&](int t) {
            const uint32_t gg = g + (uint32_t)t, s = gg % kSlots;
            if (gg >= kSlots) wait_bar(&sh.bar_slot_free[s], ((gg / kSlots) - 1) & 1, sh);
            load_rows(str_map, slots + s * slot_bytes, kTileRows, t * kTileRows, unit, &sh.bar_slot[s]);
          };
          // the first tile's slot frees before the resident chunks do
          const int pre = min(kSlots - 1, nt);
          for (int t = 0; t < pre; ++t) load_tile(t);
          for (int c = 0; c < nt; ++c) {
            if (phase > 0) wait_bar(&sh.bar_res_free[c], (phase - 1) & 1, sh);
            load_rows(res_map, res + (size_t)c * kTileRows * 16, Rr, c * kTileRows, unit, &sh.bar_res[c]);
          }
          for (int t = pre; t < nt; ++t) load_tile(t);
          g += (uint32_t)nt;
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issue
    // The whole warp walks the schedule (uniform control flow, so the
    // descriptors stay warp-uniform); one elected lane issues MMAs and commits.
    // descriptors: K-major core matrices, 8-row groups 128 B apart; the A
    // tile's K-adjacent core matrices are 128 rows apart, the resident B's Rr
    const uint32_t hi = ptx::smem_desc_hi(128);
    const uint32_t a_lo0 = ptx::smem_desc_lo(ptx::smem_addr(slots), kTileRows * 16);
    const uint32_t b_lo0 = ptx::smem_desc_lo(ptx::smem_addr(res), (uint32_t)Rr * 16);
    const uint32_t a_ks = (2 * kTileRows * 16) >> 4, b_ks = (2u * Rr * 16) >> 4;  // one K-step of 16
    const uint32_t slot_step = (uint32_t)(slot_bytes >> 4), chunk_step = (kBufCols * 16) >> 4;
    const uint32_t idesc_full = ptx::idesc_bf16_f32(kTileRows, kBufCols);
    const int nch = (a.Np + kBufCols - 1) / kBufCols;  // chunks of kBufCols keys (queries) per tile
    const uint32_t idesc_last = ptx::idesc_bf16_f32(kTileRows, a.Np - kBufCols * (nch - 1));
    const int ks_steps = a.ks_steps;
    uint32_t u = 0, g = 0, phase = 0;  // chunks, streamed tiles, passes
    for (int unit = blockIdx.x; unit < a.units; unit += gridDim.x) {
      for (int pass = 0; pass < 2; ++pass, ++phase) {
        for (int t = 0; t < nt; ++t, ++g) {
          const uint32_t s = g % kSlots;
          wait_bar(&sh.bar_slot[s], (g / kSlots) & 1, sh);
          const uint32_t a_lo = a_lo0 + s * slot_step;
          for (int c = 0; c < nch; ++c, ++u) {
            const uint32_t b = u % kBufs;
            const int p0 = c * kPieces, p1 = min(nt, p0 + kPieces);  // resident pieces of this chunk
            if (t == 0)
              for (int pc = p0; pc < p1; ++pc) wait_bar(&sh.bar_res[pc], phase & 1, sh);
            if (u >= kBufs) wait_bar(&sh.bar_empty[b], ((u / kBufs) - 1) & 1, sh);
            ptx::tc_fence_after();
            const uint32_t idesc = c == nch - 1 ? idesc_last : idesc_full;
            const uint32_t d_t = tbase + b * kBufCols;
            const uint32_t b_lo = b_lo0 + (uint32_t)c * chunk_step;
            if (ptx::elect_one()) {
              if (ks_steps == 4) mma_chunk<4>(d_t, a_lo, b_lo, hi, a_ks, b_ks, idesc);
              else if (ks_steps == 5) mma_chunk<5>(d_t, a_lo, b_lo, hi, a_ks, b_ks, idesc);
              else mma_chunk<8>(d_t, a_lo, b_lo, hi, a_ks, b_ks, idesc);
              ptx::mma_commit(&sh.bar_full[b]);
              if (t == nt - 1)
                for (int pc = p0; pc < p1; ++pc) ptx::mma_commit(&sh.bar_res_free[pc]);
            }
            __syncwarp();
          }
          if (ptx::elect_one()) ptx::mma_commit(&sh.bar_slot_free[s]);
          __syncwarp();
        }
      }
    }
    if (ptx::elect_one()) ptx::mma_commit(&sh.bar_done);
    __syncwarp();
    wait_bar(&sh.bar_done, 0, sh);
  } else {
    // ------------------------------------------------ softmax warps
    // warp w reads TMEM lane quarter (w & 3) -- the hardware ties a warp to the
    // lanes 32 * (w % 4) .. + 31 -- and its slice p = w >> 2 is the columns
    // [p * kWarpCols, + kWarpCols) of every chunk, whichever buffer holds it.
    const int quarter = warp & 3, part = warp >> 2;
    const int row = quarter * 32 + lane;
    const int col_lo = part * kWarpCols;
    const int my_cols = kWarpCols;
    const int nch = (a.Np + kBufCols - 1) / kBufCols;
    const uint32_t tlane = tbase + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col_lo;
    const float sl2 = a.sl2;
    const uint64_t sl2x2 = fm::splat2(sl2);
    float* my_part = part_lse + part * Rr;
    uint32_t u = 0;
    uint32_t v[32];
    // Runs fn(column offset) on each of the ng <= 2 32-column groups of the
    // warp's slice at TMEM address ta, the group's values in v.  One group
    // in registers at a time, straight-line: loading the second group while
    // the first is summed, or releasing the buffer before the last group's
    // arithmetic, measured slower.
    static_assert(kWarpCols <= 64, "a slice is at most two groups");
    auto for_groups = [&](uint32_t ta, int ng, auto&& fn) {
      if (ng > 0) {
        ptx::tmem_ld32(ta, v);
        ptx::tmem_wait_ld(v);
        fn(0);
      }
      if (ng > 1) {
        ptx::tmem_ld32(ta + 32, v);
        ptx::tmem_wait_ld(v);
        fn(32);
      }
    };
    // chunk u sits in buffer u % kBufs
    auto chunk_begin = [&]() {
      wait_bar(&sh.bar_full[u % kBufs], (u / kBufs) & 1, sh);
      ptx::tc_fence_after();
      return tlane + (u % kBufs) * kBufCols;
    };
    auto chunk_end = [&]() {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&sh.bar_empty[u % kBufs]);
    };
    for (int unit = blockIdx.x; unit < a.units; unit += gridDim.x) {
      // pass 1: per-part row log-sum-exp (log2 domain)
      for (int t = 0; t < nt; ++t) {
        const bool live = t * kTileRows + quarter * 32 < a.N;
        float m = -INFINITY;
        uint64_t l2 = 0;  // running sum of the row's exps, two halves
        for (int c = 0; c < nch; ++c, ++u) {
          const uint32_t taddr = chunk_begin();
          const int nc = min(my_cols, a.Np - kBufCols * c - col_lo);
          for_groups(taddr, live && nc > 0 ? nc >> 5 : 0, [&](int g) {
            const int key0 = kBufCols * c + col_lo + g;
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
            // (a group always holds a key below N, so m is finite after the
            // first group and the exps below never see m = -inf)
            if (cms > m + 8.0f) {
              l2 = fm::mul2(l2, fm::splat2(fm::ex2_mufu(m - cms)));
              m = cms;
            }
            const uint64_t nmn = fm::splat2(-m);
#pragma unroll
            for (int pr = 0; pr < 16; ++pr) {
              const uint64_t x = fm::fma2(fm::pack2(__uint_as_float(v[2 * pr]), __uint_as_float(v[2 * pr + 1])),
                                          sl2x2, nmn);
              l2 = fm::add2(l2, fm::exp2_mufu2(x));
            }
          });
          chunk_end();
        }
        float l0, l1;
        fm::unpack2(l2, l0, l1);
        my_part[t * kTileRows + row] = m == -INFINITY ? -INFINITY : m + __log2f(l0 + l1);
      }
      softmax_bar();
      for (int r = threadIdx.x; r < Rr; r += kSoftWarps * 32) {
        float M = -INFINITY;
#pragma unroll
        for (int p = 0; p < kParts; ++p) M = fmaxf(M, part_lse[p * Rr + r]);
        float L = 0.f;
#pragma unroll
        for (int p = 0; p < kParts; ++p) {
          const float lp = part_lse[p * Rr + r];
          if (lp != -INFINITY) L += fm::ex2_mufu(lp - M);
        }
        // stored negated: pass 2 adds it with one packed FMA; padded queries
        // get -inf and contribute nothing
        nlse2[r] = r < a.N ? -(M + __log2f(L)) : -INFINITY;
      }
      softmax_bar();
      // pass 2: column sums of exp2(z - lse), one key per TMEM lane
      for (int t = 0; t < nt; ++t) {
        const bool live = t * kTileRows + quarter * 32 < a.N;
        uint64_t acc = 0;
        for (int c = 0; c < nch; ++c, ++u) {
          const uint32_t taddr = chunk_begin();
          const int nc = min(my_cols, a.Np - kBufCols * c - col_lo);
          for_groups(taddr, live && nc > 0 ? nc >> 5 : 0, [&](int g) {
            // lse of the group's 32 queries: the same for every lane (broadcast
            // 16-byte loads; the offset is a multiple of 32 floats)
            const ulonglong2* nl = reinterpret_cast<const ulonglong2*>(nlse2 + kBufCols * c + col_lo + g);
#pragma unroll
            for (int pq = 0; pq < 8; ++pq) {
              const ulonglong2 w = nl[pq];
              const uint64_t x0 = fm::fma2(fm::pack2(__uint_as_float(v[4 * pq]), __uint_as_float(v[4 * pq + 1])),
                                           sl2x2, w.x);
              acc = fm::add2(acc, fm::exp2_mufu2(x0));
              const uint64_t x1 = fm::fma2(fm::pack2(__uint_as_float(v[4 * pq + 2]), __uint_as_float(v[4 * pq + 3])),
                                           sl2x2, w.y);
              acc = fm::add2(acc, fm::exp2_mufu2(x1));
            }
          });
          chunk_end();
        }
        float s0, s1;
        fm::unpack2(acc, s0, s1);
        my_part[t * kTileRows + row] = s0 + s1;
      }
      softmax_bar();
      for (int r = threadIdx.x; r < a.N; r += kSoftWarps * 32) {
        float tot = 0.f;
#pragma unroll
        for (int p = 0; p < kParts; ++p) tot += part_lse[p * Rr + r];
        a.colsum[(size_t)unit * a.N + r] = tot;
      }
      softmax_bar();  // the partials are rewritten by the next unit's pass 1
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sh.abort_flag) flag_status(a.status, kStatusTimeout);
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tbase, kTmemCols);
  }
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

// s[b][j] = inv * sum_h colsum[b][h][j], heads summed in order (inv = 1 / (H N)
// for the full salience, 1 / (H R) for the summary-row salience).
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

cudaError_t launch_head_mean(const float* colsum, int B, int H, int N, float inv, float* out,
                             cudaStream_t stream) {
  const long long total = (long long)B * N;
  if (total == 0) return cudaSuccess;
  salience_head_mean_kernel<<<(unsigned)((total + 255) / 256), 256, 0, stream>>>(colsum, B, H, N, inv, out);
  return cudaGetLastError();
}

size_t salience_smem_bytes(int N, int d) { return launch_smem(sal_geom(N, d)); }

size_t salience_workspace_bytes(int B, int H, int N, int d) {
  (void)d;
  return (size_t)B * H * N * sizeof(float);
}

cudaError_t launch_salience(const void* q, const void* k, int B, int H, int N, int d, float scale,
                            float* salience, void* ws, int* status, int num_sms,
                            cudaStream_t stream) {
  const SalGeom g = sal_geom(N, d);
  if (g.nt > kMaxChunks) return cudaErrorInvalidValue;
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
  a.units = B * H;
  a.sl2 = scale * kLog2e;
  a.colsum = static_cast<float*>(ws);
  a.status = status;
  const size_t smem = launch_smem(g);
  cudaError_t e = cudaFuncSetAttribute(salience_colsum_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = a.units < num_sms ? a.units : num_sms;
  salience_colsum_kernel<<<grid, kThreads, smem, stream>>>(tq, tk, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_head_mean(a.colsum, B, H, N, 1.0f / ((float)H * (float)N), salience, stream);
}

}  // namespace sv
