// Query-agnostic prefill salience on the tcgen05 tensor cores.
//
// velog.io SparseVILA summary §3.1: for encoders without a summary token
// (SigLIP, QwenVL) a token's salience is the intra-visual attention it
// receives, averaged over all tokens; the kernel paragraph streams the softmax
// normalisation and the salience accumulation without materialising the
// N x N attention matrix, up to hundreds of thousands of tokens.  xllm-io
// review §三 gives the formula.  Per frame b:
//   s[b][j] = 1/(H N) sum_h sum_i exp(scale q_i.k_j - lse_i),
//   lse_i   = log sum_j exp(scale q_i.k_j).
//
// Two passes per (frame, head), both on 128-row x 256-column tensor-core
// tiles (M=128, N<=256, K=16 tcgen05.mma, bf16 operands, fp32 accumulators in
// two 256-column TMEM buffers):
//   pass 1  S = Q K^T with one query per TMEM lane: each softmax thread sums
//           exp2 of its row over a 64-column slice of every chunk; the four
//           slice sums of a row give l_i and lse2_i = log2 l_i.
//   pass 2  S^T = K Q^T with one key per TMEM lane: the column sum over
//           queries becomes a per-thread row sum of exp2(z - lse2_i).
//
// -lse is folded into the pass-2 MMA: every operand row carries a 16-column
// tail K-step; the streamed (A) side holds the constants (1, 1, 1) there and
// the query (B) side the bf16 hi / mid / lo split of -lse2_i / (scale log2 e),
// so the accumulator already holds z - lse2_i / (scale log2 e) and the softmax
// threads do one multiply, one exp2 and one add per element (no lse loads).
// Padded queries carry -2^100 and contribute exactly 0.
//
// Pass 1 sums exp2 of the raw scaled logits (no running max: fp32 sums are
// scale-free, and the max tree was a third of the per-element instructions).
// A row whose sum leaves [2^-90, 2^100] (an exp overflowed, or every term
// underflowed) marks its unit in a failure list, and a second launch of the
// kernel in its exact form (a stale running max, rescaled when it grows by
// more than 8) redoes the listed units; normally the list is empty and that
// launch returns at once.
//
// Two schedules:
//   short  (N up to ~1K): persistent CTAs walk (frame, head) units; one
//          operand of a head stays resident in shared memory (K in pass 1, Q
//          in pass 2) while 128-row tiles of the other are streamed, and the
//          resident operand is replaced 128 rows at a time as the last tile
//          releases them, so the tensor pipe never drains between passes.
//   long   (any N): one launch per pass; a unit is one 128-row tile of one
//          head that stays resident while 256-row chunks of the other operand
//          stream through a ring (each chunk is reused by the tile's 128 rows:
//          128 FLOP per shared-memory byte).  Pass 1 writes each query's
//          16-byte fold record to the workspace; pass 2 loads it by TMA next to
//          the query rows.
//
// Operands sit in shared memory in the layouts the MMA reads: 64-column
// blocks in the 128-byte swizzled K-major layout (one TMA box per 128 rows),
// then the tail as 8-column no-swizzle core-matrix blocks (head-dim columns
// past the last 64-column block, then the fold column, then zeros).  Rows
// past N are zero-filled by TMA.  Head dims: 64, 72, 80, 128.
// Per-head column sums go to the workspace; a second kernel averages heads in
// a fixed order (deterministic).
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "fastmath.cuh"
#include "tc_ptx.cuh"

namespace sv {

namespace {

constexpr int kBufs = 2;                       // TMEM buffers (one chunk each)
constexpr int kBufCols = 256;                  // columns of one TMEM buffer (N of one MMA)
constexpr int kSlices = 4;                     // softmax warps per TMEM lane quarter
constexpr int kWarpCols = kBufCols / kSlices;  // columns of every chunk per softmax warp
static_assert(kWarpCols == 64, "a slice is two 32-column groups");
constexpr int kParts = kSlices;                // row partials per lane (one per slice)
constexpr int kSoftWarps = 4 * kSlices;
constexpr int kMmaWarp = kSoftWarps, kTmaWarp = kSoftWarps + 1;
constexpr int kThreads = (kSoftWarps + 2) * 32;
constexpr int kTileRows = 128;
constexpr int kChunkRows = kBufCols;
constexpr int kTmemCols = 512;
static_assert(kBufs * kBufCols <= kTmemCols, "TMEM buffers exceed the allocation");
constexpr int kSlots = 2;        // short schedule: streamed 128-row tiles in flight
constexpr int kMaxPieces = 8;    // short schedule: resident 128-row pieces (N <= 1024)
constexpr int kAStages = 2;      // long schedule: resident tiles
constexpr int kMaxBStages = 3;   // long schedule: streamed chunks
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr size_t kMaxDynSmem = 232448;
constexpr float kFoldPad = -1.2676506002282294e30f;  // -2^100
constexpr float kSumLo = 8.0779356694631609e-28f;    // 2^-90
constexpr float kSumHi = 1.2676506002282294e30f;     // 2^100
constexpr float kMaskLogit = -1.0e30f;               // keys past N in pass 1

enum Sched { kShort = 0, kLongRows = 1, kLongCols = 2 };

// Shared-memory geometry of one operand row for head dim d = 64 MB + 8 TD.
template <int MB, int TD>
struct Geo {
  static constexpr int kTailSteps = (TD + 2) / 2;   // tail K-steps: data, fold (+ zero) blocks
  static constexpr int kTailCms = 2 * kTailSteps;   // 8-column core-matrix blocks in the tail
  static constexpr int kFoldCm = TD;
  static constexpr int kRowBytes = 128 * MB + 16 * kTailCms;
  // byte offsets inside a buffer of R rows
  static __host__ __device__ constexpr uint32_t main_off(int R, int b) { return (uint32_t)b * R * 128u; }
  static __host__ __device__ constexpr uint32_t tail_off(int R, int i) {
    return (uint32_t)MB * R * 128u + (uint32_t)i * R * 16u;
  }
  static constexpr uint32_t kTmaBytes128 = 128u * (128u * MB + 16u * TD);  // one 128-row load
};

struct SalArgs {
  int N, Np, nt, nch;   // tokens, N rounded up to 32, 128-row tiles, 256-column chunks
  int Rr;               // short schedule: resident rows (nt * 128)
  int units;            // short: B*H; long: B*H*nt
  int Nf;               // long schedule: fold records per head (>= nch * 256)
  int bstages;          // long schedule: streamed chunks in flight
  int list_mode;        // 1: the units come from the failure list
  float sl2, inv_sl2;   // scale * log2(e) and its inverse
  float* colsum;        // [B*H][N]
  uint4* fold;          // long schedule: [B*H][Nf] fold records
  int* fail_count;      // failure list length (reset by the list launch)
  int* fail_done;       // CTAs of the list launch that have finished
  int* fail_list;
  int* status;
};

struct SalShared {
  uint64_t bar_done, bar_lse;
  uint64_t bar_full[kBufs], bar_empty[kBufs];
  uint64_t bar_in[kMaxPieces], bar_in_free[kMaxPieces];     // resident pieces / tile stages
  uint64_t bar_st[kMaxBStages], bar_st_free[kMaxBStages];   // streamed tiles / chunk stages
  uint32_t tmem_base;
  int abort_flag;
  int unit_fail;
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

__device__ __forceinline__ void softmax_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kSoftWarps * 32) : "memory"); }

// 16-byte fold record: bf16 (hi, mid, lo) with hi + mid + lo == v exactly
// (each remainder is exact in fp32), then zeros.
__device__ __forceinline__ uint4 fold_record(float v) {
  const uint32_t h = f32_to_bf16_bits(v);
  const float r1 = v - __uint_as_float(h << 16);
  const uint32_t m = f32_to_bf16_bits(r1);
  const float r2 = r1 - __uint_as_float(m << 16);
  const uint32_t l = f32_to_bf16_bits(r2);
  return make_uint4(h | (m << 16), l, 0u, 0u);
}
constexpr uint32_t kBf16One = 0x3f80u;
__device__ __forceinline__ uint4 ones_record() { return make_uint4(kBf16One | (kBf16One << 16), kBf16One, 0u, 0u); }

// Fills rows [0, R) of tail block i of the buffer at `buf` with `val`
// (threads tid0, tid0 + nthr, ...).
template <class G>
__device__ __forceinline__ void fill_tail(uint8_t* buf, int R, int i, uint4 val, int tid0, int nthr) {
  uint4* p = reinterpret_cast<uint4*>(buf + G::tail_off(R, i));
  for (int r = tid0; r < R; r += nthr) p[r] = val;
}

// 128 rows of one head: the 64-column blocks (swizzled) and the tail data
// blocks, into rows [dst_row0, +128) of a buffer of R rows.
template <class G, int MB, int TD>
__device__ __forceinline__ void tma_rows(const CUtensorMap* main_map, const CUtensorMap* tail_map, uint8_t* buf,
                                         int R, int dst_row0, int row0, int head, uint64_t* bar) {
#pragma unroll
  for (int b = 0; b < MB; ++b)
    ptx::tma_load_3d(buf + G::main_off(R, b) + (uint32_t)dst_row0 * 128u, main_map, 64 * b, row0, head, bar);
#pragma unroll
  for (int i = 0; i < TD; ++i)
    ptx::tma_load_3d(buf + G::tail_off(R, i) + (uint32_t)dst_row0 * 16u, tail_map, 64 * MB + 8 * i, row0, head,
                     bar);
}

// KS K-steps of one 128 x n chunk: A rows [0, 128) of a buffer of RA rows, B
// rows [rb0, rb0 + n) of a buffer of RB rows.
template <class G, int MB>
__device__ __forceinline__ void mma_chunk(uint32_t d_t, uint32_t a_base, int RA, uint32_t b_base, int RB, int rb0,
                                          uint32_t idesc) {
  const uint32_t hi_sw = ptx::smem_desc_hi_sw128(1024);
  const uint32_t hi_ns = ptx::smem_desc_hi(128);
#pragma unroll
  for (int k = 0; k < 4 * MB; ++k) {
    const uint32_t a = ptx::smem_desc_lo_sw128(a_base + G::main_off(RA, k / 4) + (uint32_t)(k % 4) * 32u);
    const uint32_t b =
        ptx::smem_desc_lo_sw128(b_base + G::main_off(RB, k / 4) + (uint32_t)rb0 * 128u + (uint32_t)(k % 4) * 32u);
    ptx::mma_bf16_split(d_t, a, b, hi_sw, idesc, k > 0 ? 1u : 0u);
  }
#pragma unroll
  for (int s = 0; s < G::kTailSteps; ++s) {
    const uint32_t a = ptx::smem_desc_lo(a_base + G::tail_off(RA, 2 * s), (uint32_t)RA * 16u);
    const uint32_t b = ptx::smem_desc_lo(b_base + G::tail_off(RB, 2 * s) + (uint32_t)rb0 * 16u, (uint32_t)RB * 16u);
    ptx::mma_bf16_split(d_t, a, b, hi_ns, idesc, 1u);
  }
}

// Dynamic shared memory of one schedule (before the 1 KB alignment slack).
template <int MB, int TD>
size_t smem_need(int sched, int Rr, int bstages) {
  using G = Geo<MB, TD>;
  if (sched == kShort)
    return (size_t)Rr * G::kRowBytes + (size_t)kSlots * kTileRows * G::kRowBytes + (size_t)kParts * Rr * 4;
  return (size_t)kAStages * kTileRows * G::kRowBytes + (size_t)bstages * kChunkRows * G::kRowBytes +
         (size_t)kParts * kTileRows * 4;
}

template <int MB, int TD, int SCHED, bool EXACT>
__global__ void __launch_bounds__(kThreads, 1)
salience_kernel(const __grid_constant__ CUtensorMap tq_main, const __grid_constant__ CUtensorMap tq_tail,
                const __grid_constant__ CUtensorMap tk_main, const __grid_constant__ CUtensorMap tk_tail,
                const __grid_constant__ CUtensorMap tf, SalArgs a) {
  using G = Geo<MB, TD>;
  constexpr bool kShortS = SCHED == kShort;
  extern __shared__ uint8_t smem_raw[];
  __shared__ SalShared sh;

  // the exact re-run only takes units from the failure list (normally empty)
  int n_units = a.units;
  if (a.list_mode) {
    n_units = *(volatile int*)a.fail_count;
    if ((int)blockIdx.x >= n_units) return;
  }

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int nt = a.nt, nch = a.nch;
  // short: resident [Rr rows] | kSlots streamed tiles [128 rows] | partials [kParts][Rr]
  // long:  kAStages resident tiles [128 rows] | bstages chunks [256 rows] | partials [kParts][128]
  const int R_in = kShortS ? a.Rr : kTileRows;                  // rows of one "in" buffer (the B side in short)
  const int n_in = kShortS ? 1 : kAStages;
  const int R_st = kShortS ? kTileRows : kChunkRows;            // rows of one streamed buffer
  const int n_st = kShortS ? kSlots : a.bstages;
  uint8_t* in_base = smem;
  uint8_t* st_base = smem + (size_t)n_in * R_in * G::kRowBytes;
  float* part = reinterpret_cast<float*>(st_base + (size_t)n_st * R_st * G::kRowBytes);
  const int PR = kShortS ? a.Rr : kTileRows;                    // rows of one partials array
  auto in_buf = [&](int i) { return in_base + (size_t)i * R_in * G::kRowBytes; };
  auto st_buf = [&](int i) { return st_base + (size_t)i * R_st * G::kRowBytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Tail blocks TMA never writes.  The streamed tiles of the short schedule
  // and the resident tile of the long one carry the MMA's side of the fold
  // (ones); the other side starts at zero (short: rewritten per unit; long
  // pass 1: zero; long pass 2: fold records loaded by TMA).
  for (int i = TD; i < G::kTailCms; ++i) {
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const bool fold = i == G::kFoldCm;
    if (kShortS) {
      fill_tail<G>(in_buf(0), R_in, i, zero, threadIdx.x, blockDim.x);
      for (int s = 0; s < n_st; ++s) fill_tail<G>(st_buf(s), R_st, i, fold ? ones_record() : zero, threadIdx.x, blockDim.x);
    } else {
      for (int s = 0; s < n_in; ++s) fill_tail<G>(in_buf(s), R_in, i, fold ? ones_record() : zero, threadIdx.x, blockDim.x);
      if (!(fold && SCHED == kLongCols))
        for (int s = 0; s < n_st; ++s) fill_tail<G>(st_buf(s), R_st, i, zero, threadIdx.x, blockDim.x);
    }
  }
  ptx::fence_proxy_async_smem();

  if (threadIdx.x == 0) {
    ptx::mbar_init(&sh.bar_done, 1);
    ptx::mbar_init(&sh.bar_lse, 1);
    for (int i = 0; i < kBufs; ++i) {
      ptx::mbar_init(&sh.bar_full[i], 1);
      ptx::mbar_init(&sh.bar_empty[i], kSoftWarps);  // every softmax warp reads every chunk
    }
    for (int i = 0; i < kMaxPieces; ++i) {
      ptx::mbar_init(&sh.bar_in[i], 1);
      ptx::mbar_init(&sh.bar_in_free[i], 1);
    }
    for (int i = 0; i < kMaxBStages; ++i) {
      ptx::mbar_init(&sh.bar_st[i], 1);
      ptx::mbar_init(&sh.bar_st_free[i], 1);
    }
    sh.abort_flag = 0;
    sh.unit_fail = 0;
    ptx::mbar_fence_init();
  }
  if (warp == 0) ptx::tmem_alloc(&sh.tmem_base, kTmemCols);
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tbase = sh.tmem_base;
  auto unit_at = [&](int i) { return a.list_mode ? __ldcg(a.fail_list + i) : i; };

  if (warp == kTmaWarp) {
    // ------------------------------------------------ TMA loads (lane 0 issues)
    if (lane == 0) {
      ptx::prefetch_tensormap(&tq_main);
      ptx::prefetch_tensormap(&tk_main);
      if (TD > 0) {
        ptx::prefetch_tensormap(&tq_tail);
        ptx::prefetch_tensormap(&tk_tail);
      }
      if (SCHED == kLongCols) ptx::prefetch_tensormap(&tf);
    }
    if (kShortS) {
      uint32_t g = 0, phase = 0;  // streamed tiles, passes issued so far
      for (int i = blockIdx.x; i < n_units; i += gridDim.x) {
        const int head = unit_at(i);
        for (int pass = 0; pass < 2; ++pass, ++phase) {
          const CUtensorMap* res_main = pass == 0 ? &tk_main : &tq_main;
          const CUtensorMap* res_tail = pass == 0 ? &tk_tail : &tq_tail;
          const CUtensorMap* str_main = pass == 0 ? &tq_main : &tk_main;
          const CUtensorMap* str_tail = pass == 0 ? &tq_tail : &tk_tail;
          auto load_tile = [&](int t) {
            const uint32_t gg = g + (uint32_t)t, s = gg % kSlots;
            if (gg >= kSlots) wait_bar(&sh.bar_st_free[s], ((gg / kSlots) - 1) & 1, sh);
            if (lane == 0) {
              ptx::mbar_arrive_expect_tx(&sh.bar_st[s], G::kTmaBytes128);
              tma_rows<G, MB, TD>(str_main, str_tail, st_buf(s), R_st, 0, t * kTileRows, head, &sh.bar_st[s]);
            }
            __syncwarp();
          };
          // the first tile's slot frees before the resident pieces do
          const int pre = min(kSlots - 1, nt);
          for (int t = 0; t < pre; ++t) load_tile(t);
          for (int c = 0; c < nt; ++c) {
            if (phase > 0) wait_bar(&sh.bar_in_free[c], (phase - 1) & 1, sh);
            if (pass == 0) {
              // keys carry no fold: clear the previous unit's records on this piece
              uint4* f = reinterpret_cast<uint4*>(in_buf(0) + G::tail_off(R_in, G::kFoldCm)) + c * kTileRows;
              for (int r = lane; r < kTileRows; r += 32) f[r] = make_uint4(0u, 0u, 0u, 0u);
              ptx::fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) {
              ptx::mbar_arrive_expect_tx(&sh.bar_in[c], G::kTmaBytes128);
              tma_rows<G, MB, TD>(res_main, res_tail, in_buf(0), R_in, c * kTileRows, c * kTileRows, head,
                                  &sh.bar_in[c]);
            }
            __syncwarp();
          }
          for (int t = pre; t < nt; ++t) load_tile(t);
          g += (uint32_t)nt;
        }
      }
    } else {
      const CUtensorMap* in_main = SCHED == kLongRows ? &tq_main : &tk_main;
      const CUtensorMap* in_tail = SCHED == kLongRows ? &tq_tail : &tk_tail;
      const CUtensorMap* st_main = SCHED == kLongRows ? &tk_main : &tq_main;
      const CUtensorMap* st_tail = SCHED == kLongRows ? &tk_tail : &tq_tail;
      const uint32_t chunk_bytes = 2u * G::kTmaBytes128 + (SCHED == kLongCols ? kChunkRows * 16u : 0u);
      const int S = a.bstages;
      uint32_t j = 0, v = 0;  // units, chunks issued so far
      for (int i = blockIdx.x; i < n_units; i += gridDim.x, ++j) {
        const int unit = unit_at(i);
        const int head = unit / nt, t = unit % nt;
        const uint32_t as = j % kAStages;
        if (j >= kAStages) wait_bar(&sh.bar_in_free[as], ((j / kAStages) - 1) & 1, sh);
        if (lane == 0) {
          ptx::mbar_arrive_expect_tx(&sh.bar_in[as], G::kTmaBytes128);
          tma_rows<G, MB, TD>(in_main, in_tail, in_buf(as), R_in, 0, t * kTileRows, head, &sh.bar_in[as]);
        }
        __syncwarp();
        for (int c = 0; c < nch; ++c, ++v) {
          const uint32_t s = v % S;
          if (v >= (uint32_t)S) wait_bar(&sh.bar_st_free[s], ((v / S) - 1) & 1, sh);
          if (lane == 0) {
            ptx::mbar_arrive_expect_tx(&sh.bar_st[s], chunk_bytes);
            for (int h = 0; h < 2; ++h) {
              const int row0 = c * kChunkRows + h * kTileRows;
              tma_rows<G, MB, TD>(st_main, st_tail, st_buf(s), R_st, h * kTileRows, row0, head, &sh.bar_st[s]);
              if (SCHED == kLongCols)
                ptx::tma_load_3d(st_buf(s) + G::tail_off(R_st, G::kFoldCm) + (uint32_t)h * kTileRows * 16u, &tf, 0,
                                 row0, head, &sh.bar_st[s]);
            }
          }
          __syncwarp();
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------ MMA issue
    // The whole warp walks the schedule (uniform control flow); one elected
    // lane issues MMAs and commits.
    const uint32_t idesc_full = ptx::idesc_bf16_f32(kTileRows, kBufCols);
    const uint32_t idesc_last = ptx::idesc_bf16_f32(kTileRows, a.Np - kBufCols * (nch - 1));
    uint32_t u = 0;  // chunks issued (TMEM buffer u % kBufs)
    auto issue = [&](uint8_t* abuf, int RA, uint8_t* bbuf, int RB, int rb0, int c) {
      const uint32_t b = u % kBufs;
      if (u >= kBufs) wait_bar(&sh.bar_empty[b], ((u / kBufs) - 1) & 1, sh);
      ptx::tc_fence_after();
      if (ptx::elect_one()) {
        mma_chunk<G, MB>(tbase + b * kBufCols, ptx::smem_addr(abuf), RA, ptx::smem_addr(bbuf), RB, rb0,
                         c == nch - 1 ? idesc_last : idesc_full);
        ptx::mma_commit(&sh.bar_full[b]);
      }
      __syncwarp();
      ++u;
    };
    if (kShortS) {
      uint32_t g = 0, phase = 0, j = 0;  // streamed tiles, passes, units
      for (int i = blockIdx.x; i < n_units; i += gridDim.x, ++j) {
        for (int pass = 0; pass < 2; ++pass, ++phase) {
          // pass 2 reads the queries' fold records
          if (pass == 1) wait_bar(&sh.bar_lse, j & 1, sh);
          for (int t = 0; t < nt; ++t, ++g) {
            const uint32_t s = g % kSlots;
            wait_bar(&sh.bar_st[s], (g / kSlots) & 1, sh);
            for (int c = 0; c < nch; ++c) {
              const int p0 = c * (kChunkRows / kTileRows), p1 = min(nt, p0 + kChunkRows / kTileRows);
              if (t == 0)
                for (int pc = p0; pc < p1; ++pc) wait_bar(&sh.bar_in[pc], phase & 1, sh);
              issue(st_buf(s), R_st, in_buf(0), R_in, c * kChunkRows, c);
              if (t == nt - 1) {
                if (ptx::elect_one())
                  for (int pc = p0; pc < p1; ++pc) ptx::mma_commit(&sh.bar_in_free[pc]);
                __syncwarp();
              }
            }
            if (ptx::elect_one()) ptx::mma_commit(&sh.bar_st_free[s]);
            __syncwarp();
          }
        }
      }
    } else {
      const int S = a.bstages;
      uint32_t j = 0, v = 0;
      for (int i = blockIdx.x; i < n_units; i += gridDim.x, ++j) {
        const uint32_t as = j % kAStages;
        wait_bar(&sh.bar_in[as], (j / kAStages) & 1, sh);
        for (int c = 0; c < nch; ++c, ++v) {
          const uint32_t s = v % S;
          wait_bar(&sh.bar_st[s], (v / S) & 1, sh);
          issue(in_buf(as), R_in, st_buf(s), R_st, 0, c);
          if (ptx::elect_one()) ptx::mma_commit(&sh.bar_st_free[s]);
          __syncwarp();
        }
        if (ptx::elect_one()) ptx::mma_commit(&sh.bar_in_free[as]);
        __syncwarp();
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
    const int quarter = warp & 3, slice = warp >> 2;
    const int row = quarter * 32 + lane;
    const int col_lo = slice * kWarpCols;
    const uint32_t tlane = tbase + ((uint32_t)(quarter * 32) << 16) + (uint32_t)col_lo;
    const uint64_t sl2x2 = fm::splat2(a.sl2);
    const int tid = threadIdx.x;
    float* my_part = part + slice * PR;
    uint32_t u = 0;
    uint32_t v[32];

    // One 128-row tile against every chunk: fn(chunk, group column offset,
    // registers) on each 32-column group of the warp's slice, one group in
    // registers at a time (a single 64-column load, or releasing the buffer
    // before the math, measured slower).
    // Every chunk but the last has 256 columns (two groups per slice, no key
    // past N); the last chunk's group count per slice is fixed per launch.
    static_assert(kBufs == 2, "the chunk counter's low bit is the buffer");
    const int nc_last = min(kWarpCols, a.Np - kBufCols * (nch - 1) - col_lo);
    const int ng_last = nc_last > 0 ? nc_last >> 5 : 0;
    auto run_tile = [&](bool live, auto&& fn) {
      auto chunk = [&](int c, int ng, bool last) {
        const uint32_t b = u & 1u;
        wait_bar(&sh.bar_full[b], (u >> 1) & 1u, sh);
        ptx::tc_fence_after();
        const uint32_t taddr = tlane + b * kBufCols;
        if (ng > 0) {
          ptx::tmem_ld32(taddr, v);
          ptx::tmem_wait_ld(v);
          fn(c, 0, v, last);
        }
        if (ng > 1) {
          ptx::tmem_ld32(taddr + 32, v);
          ptx::tmem_wait_ld(v);
          fn(c, 32, v, last);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sh.bar_empty[b]);
        ++u;
      };
      const int ng_full = live ? 2 : 0;
      for (int c = 0; c < nch - 1; ++c) chunk(c, ng_full, false);
      chunk(nch - 1, live ? ng_last : 0, true);
    };
    // sum of exp2(sl2 * r) over a group, into the packed accumulator (all on
    // MUFU: moving a share of the exps to an FMA-pipe polynomial measured
    // slower -- the softmax warps are latency-bound, not MUFU-queue-bound)
    auto sum_exp = [&](uint64_t& acc, const uint32_t* r) {
#pragma unroll
      for (int pr = 0; pr < 16; ++pr)
        acc = fm::add2(acc, fm::exp2_mufu2(fm::mul2(fm::pack2(__uint_as_float(r[2 * pr]),
                                                              __uint_as_float(r[2 * pr + 1])), sl2x2)));
    };
    // keys >= N (zero rows from TMA) contribute nothing in pass 1
    auto mask_keys = [&](int key0, uint32_t* r) {
      if (key0 + 32 > a.N) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (key0 + i >= a.N) r[i] = __float_as_uint(kMaskLogit);
      }
    };
    // pass 1 of one tile: the row's partial sum over this slice (optimistic),
    // or its partial log2-sum-exp (exact: stale running max, MUFU only)
    auto tile_rows = [&](int t) -> float {
      const bool live = t * kTileRows + quarter * 32 < a.N;
      if (!EXACT) {
        uint64_t acc = 0;
        run_tile(live, [&](int c, int gofs, uint32_t* r, bool last) {
          if (last) mask_keys(kBufCols * c + col_lo + gofs, r);
          sum_exp(acc, r);
        });
        float l0, l1;
        fm::unpack2(acc, l0, l1);
        return l0 + l1;
      } else {
        float m = -INFINITY;
        uint64_t l2 = 0;
        run_tile(live, [&](int c, int gofs, uint32_t* r, bool last) {
          if (last) mask_keys(kBufCols * c + col_lo + gofs, r);
          float mx[11];
#pragma unroll
          for (int i = 0; i < 10; ++i)
            mx[i] = fm::max3(__uint_as_float(r[3 * i]), __uint_as_float(r[3 * i + 1]), __uint_as_float(r[3 * i + 2]));
          mx[10] = fmaxf(__uint_as_float(r[30]), __uint_as_float(r[31]));
          const float cm = fmaxf(fm::max3(fm::max3(mx[0], mx[1], mx[2]), fm::max3(mx[3], mx[4], mx[5]),
                                          fm::max3(mx[6], mx[7], mx[8])),
                                 fmaxf(mx[9], mx[10]));
          // stale running max: rescale only when the group max exceeds it by
          // more than 8 (log2 units); a group always holds a key below N
          const float cms = cm * a.sl2;
          if (cms > m + 8.0f) {
            l2 = fm::mul2(l2, fm::splat2(fm::ex2_mufu(m - cms)));
            m = cms;
          }
          const uint64_t nmn = fm::splat2(-m);
#pragma unroll
          for (int pr = 0; pr < 16; ++pr) {
            const uint64_t x = fm::fma2(fm::pack2(__uint_as_float(r[2 * pr]), __uint_as_float(r[2 * pr + 1])),
                                        sl2x2, nmn);
            l2 = fm::add2(l2, fm::exp2_mufu2(x));
          }
        });
        float l0, l1;
        fm::unpack2(l2, l0, l1);
        return m == -INFINITY ? -INFINITY : m + __log2f(l0 + l1);
      }
    };
    // pass 2 of one tile: the key's partial column sum over this slice
    auto tile_cols = [&](int t) -> float {
      const bool live = t * kTileRows + quarter * 32 < a.N;
      uint64_t acc = 0;
      run_tile(live, [&](int, int, uint32_t* r, bool) { sum_exp(acc, r); });
      float s0, s1;
      fm::unpack2(acc, s0, s1);
      return s0 + s1;
    };
    // merged log2 l of row r (sum of the slices' partials); false when the
    // optimistic sum left the safe range
    auto merge_row = [&](int r, float& lse2) -> bool {
      if (!EXACT) {
        float L = 0.f;
#pragma unroll
        for (int p = 0; p < kParts; ++p) L += part[p * PR + r];
        lse2 = __log2f(L);
        return L >= kSumLo && L <= kSumHi;
      } else {
        float M = -INFINITY;
#pragma unroll
        for (int p = 0; p < kParts; ++p) M = fmaxf(M, part[p * PR + r]);
        float L = 0.f;
#pragma unroll
        for (int p = 0; p < kParts; ++p) {
          const float lp = part[p * PR + r];
          if (lp != -INFINITY) L += fm::ex2_mufu(lp - M);
        }
        lse2 = M + __log2f(L);
        return true;
      }
    };
    auto record_failure = [&](int unit) {
      if (tid == 0) {
        if (sh.unit_fail) {
          const int slot = atomicAdd(a.fail_count, 1);
          a.fail_list[slot] = unit;
          sh.unit_fail = 0;
        }
      }
    };

    if (kShortS) {
      uint4* fold_cm = reinterpret_cast<uint4*>(in_buf(0) + G::tail_off(R_in, G::kFoldCm));
      for (int i = blockIdx.x; i < n_units; i += gridDim.x) {
        const int unit = unit_at(i);
        for (int t = 0; t < nt; ++t) {
          const float p = tile_rows(t);
          my_part[t * kTileRows + row] = p;
        }
        softmax_bar();
        // fold records of the unit's queries into the resident Q rows
        for (int r = tid; r < a.Rr; r += kSoftWarps * 32) {
          float lse2 = 0.f;
          const bool ok = merge_row(r, lse2);
          if (r < a.N && !ok) sh.unit_fail = 1;
          fold_cm[r] = fold_record(r < a.N ? -lse2 * a.inv_sl2 : kFoldPad);
        }
        ptx::fence_proxy_async_smem();
        softmax_bar();
        if (tid == 0) ptx::mbar_arrive(&sh.bar_lse);
        record_failure(unit);
        for (int t = 0; t < nt; ++t) {
          const float p = tile_cols(t);
          my_part[t * kTileRows + row] = p;
        }
        softmax_bar();
        for (int r = tid; r < a.N; r += kSoftWarps * 32) {
          float tot = 0.f;
#pragma unroll
          for (int p = 0; p < kParts; ++p) tot += part[p * PR + r];
          a.colsum[(size_t)unit * a.N + r] = tot;
        }
        softmax_bar();  // the partials are rewritten by the next unit's pass 1
      }
    } else {
      for (int i = blockIdx.x; i < n_units; i += gridDim.x) {
        const int unit = unit_at(i);
        const int head = unit / nt, t = unit % nt;
        const float p = SCHED == kLongRows ? tile_rows(t) : tile_cols(t);
        my_part[row] = p;
        softmax_bar();
        if (tid < kTileRows) {
          const int r = t * kTileRows + tid;
          if (SCHED == kLongRows) {
            float lse2 = 0.f;
            const bool ok = merge_row(tid, lse2);
            if (r < a.N && !ok) sh.unit_fail = 1;
            a.fold[(size_t)head * a.Nf + r] = fold_record(r < a.N ? -lse2 * a.inv_sl2 : kFoldPad);
          } else if (r < a.N) {
            float tot = 0.f;
#pragma unroll
            for (int q = 0; q < kParts; ++q) tot += part[q * PR + tid];
            a.colsum[(size_t)head * a.N + r] = tot;
          }
        }
        softmax_bar();
        if (SCHED == kLongRows) record_failure(unit);
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0 && sh.abort_flag) flag_status(a.status, kStatusTimeout);
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tbase, kTmemCols);
  }
  // the list launch empties the list once every participating CTA is done
  if (a.list_mode && threadIdx.x == 0) {
    __threadfence();
    const int participating = min((int)gridDim.x, n_units);
    if (atomicAdd(a.fail_done, 1) == participating - 1) {
      *a.fail_count = 0;
      *a.fail_done = 0;
    }
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

// bf16 [units][rows][cols] tensor, box {box_cols, 128, 1}.
bool make_map(CUtensorMap* map, const void* base, int cols, int rows, int units, int box_cols, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)units};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)rows * cols * 2};
  cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)kTileRows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Schedule and buffer sizes of one call.
struct Plan {
  int sched;      // kShort or long
  int Rr, nt, nch, Np, Nf, bstages;
  size_t smem;    // dynamic shared memory to request
};

template <int MB, int TD>
Plan make_plan(int N) {
  using G = Geo<MB, TD>;
  Plan p;
  p.nt = (N + kTileRows - 1) / kTileRows;
  p.Np = (N + 31) / 32 * 32;
  p.nch = (p.Np + kChunkRows - 1) / kChunkRows;
  p.Rr = p.nt * kTileRows;
  p.Nf = p.nch * kChunkRows;
  p.bstages = G::kRowBytes <= 192 ? 3 : 2;
  const size_t slack = 1024 + sizeof(SalShared) + 256;
  const size_t short_need = smem_need<MB, TD>(kShort, p.Rr, 0);
  if (p.nt <= kMaxPieces && short_need + slack <= kMaxDynSmem) {
    p.sched = kShort;
    p.smem = short_need + 1024;
  } else {
    p.sched = kLongRows;
    p.smem = smem_need<MB, TD>(kLongRows, 0, p.bstages) + 1024;
  }
  // every CTA holds all 512 TMEM columns: at most one CTA per SM
  const size_t one_per_sm = 120 * 1024;
  if (p.smem < one_per_sm) p.smem = one_per_sm;
  return p;
}

// Workspace after the status word: colsum [B*H][N] | fail counters (256 B) |
// fail list [units] | long schedule: fold records [B*H][Nf].
struct WsLayout {
  size_t colsum, counters, list, fold, total;
};
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
WsLayout ws_layout(int B, int H, int N, const Plan& p) {
  WsLayout w;
  const size_t bh = (size_t)B * H;
  const size_t units = p.sched == kShort ? bh : bh * p.nt;
  w.colsum = 0;
  w.counters = round256(bh * N * sizeof(float));
  w.list = w.counters + 256;
  w.fold = w.list + round256(units * sizeof(int));
  w.total = w.fold + (p.sched == kShort ? 0 : round256(bh * p.Nf * 16));
  return w;
}

template <int MB, int TD, int SCHED, bool EXACT>
cudaError_t launch_one(const CUtensorMap* maps, const SalArgs& a, int grid, size_t smem, cudaStream_t stream) {
  auto kern = salience_kernel<MB, TD, SCHED, EXACT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, stream>>>(maps[0], maps[1], maps[2], maps[3], maps[4], a);
  return cudaGetLastError();
}

template <int MB, int TD>
Plan plan_for(int N) { return make_plan<MB, TD>(N); }

Plan plan_of(int N, int d) {
  switch (d) {
    case 64: return plan_for<1, 0>(N);
    case 72: return plan_for<1, 1>(N);
    case 80: return plan_for<1, 2>(N);
    default: return plan_for<2, 0>(N);
  }
}

template <int MB, int TD>
cudaError_t run_salience(const void* q, const void* k, int B, int H, int N, int d, float scale, float* salience,
                         void* ws, int* status, int num_sms, cudaStream_t stream) {
  const Plan p = make_plan<MB, TD>(N);
  const WsLayout w = ws_layout(B, H, N, p);
  char* base = static_cast<char*>(ws);
  const int BH = B * H;
  // maps: Q main, Q tail, K main, K tail, fold records
  CUtensorMap maps[5];
  memset(maps, 0, sizeof(maps));
  if (!make_map(&maps[0], q, d, N, BH, 64, true) || !make_map(&maps[2], k, d, N, BH, 64, true))
    return cudaErrorInvalidValue;
  if (TD > 0 && (!make_map(&maps[1], q, d, N, BH, 8, false) || !make_map(&maps[3], k, d, N, BH, 8, false)))
    return cudaErrorInvalidValue;
  if (p.sched != kShort && !make_map(&maps[4], base + w.fold, 8, p.Nf, BH, 8, false)) return cudaErrorInvalidValue;

  SalArgs a;
  a.N = N;
  a.Np = p.Np;
  a.nt = p.nt;
  a.nch = p.nch;
  a.Rr = p.Rr;
  a.Nf = p.Nf;
  a.bstages = p.bstages;
  a.list_mode = 0;
  a.sl2 = scale * kLog2e;
  a.inv_sl2 = 1.0f / a.sl2;
  a.colsum = reinterpret_cast<float*>(base + w.colsum);
  a.fold = reinterpret_cast<uint4*>(base + w.fold);
  a.fail_count = reinterpret_cast<int*>(base + w.counters);
  a.fail_done = a.fail_count + 1;
  a.fail_list = reinterpret_cast<int*>(base + w.list);
  a.status = status;
  cudaError_t e;
  if (p.sched == kShort) {
    a.units = BH;
    const int grid = BH < num_sms ? BH : num_sms;
    e = launch_one<MB, TD, kShort, false>(maps, a, grid, p.smem, stream);
    if (e != cudaSuccess) return e;
    a.list_mode = 1;   // exact re-run of the units whose row sums left the safe range
    e = launch_one<MB, TD, kShort, true>(maps, a, grid, p.smem, stream);
  } else {
    a.units = BH * p.nt;
    const int grid = a.units < num_sms ? a.units : num_sms;
    e = launch_one<MB, TD, kLongRows, false>(maps, a, grid, p.smem, stream);
    if (e != cudaSuccess) return e;
    a.list_mode = 1;
    e = launch_one<MB, TD, kLongRows, true>(maps, a, grid, p.smem, stream);
    if (e != cudaSuccess) return e;
    a.list_mode = 0;
    e = launch_one<MB, TD, kLongCols, false>(maps, a, grid, p.smem, stream);
  }
  if (e != cudaSuccess) return e;
  return launch_head_mean(a.colsum, B, H, N, 1.0f / ((float)H * (float)N), salience, stream);
}

}  // namespace

// s[b][j] = inv * sum_h colsum[b][h][j], heads summed in order (inv = 1 / (H N)
// for the full salience, 1 / (H R) for the summary-row salience).
__global__ void salience_head_mean_kernel(const float* __restrict__ colsum, int B, int H, int N,
                                          float inv, float* __restrict__ out) {
  grid_dep_sync();
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
  return launch_dependent(salience_head_mean_kernel, dim3((unsigned)((total + 255) / 256)), dim3(256), 0, stream,
                          colsum, B, H, N, inv, out);
}

bool salience_head_dim_supported(int d) { return d == 64 || d == 72 || d == 80 || d == 128; }

bool salience_uses_long_schedule(int N, int d) { return plan_of(N, d).sched != kShort; }

int salience_kernel_count(int N, int d) { return salience_uses_long_schedule(N, d) ? 4 : 3; }

size_t salience_workspace_bytes(int B, int H, int N, int d) {
  return ws_layout(B, H, N, plan_of(N, d)).total;
}

cudaError_t launch_salience(const void* q, const void* k, int B, int H, int N, int d, float scale,
                            float* salience, void* ws, int* status, int num_sms, cudaStream_t stream) {
  switch (d) {
    case 64: return run_salience<1, 0>(q, k, B, H, N, d, scale, salience, ws, status, num_sms, stream);
    case 72: return run_salience<1, 1>(q, k, B, H, N, d, scale, salience, ws, status, num_sms, stream);
    case 80: return run_salience<1, 2>(q, k, B, H, N, d, scale, salience, ws, status, num_sms, stream);
    case 128: return run_salience<2, 0>(q, k, B, H, N, d, scale, salience, ws, status, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace sv
