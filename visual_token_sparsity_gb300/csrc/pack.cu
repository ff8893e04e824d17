// Pack-once KV for round reuse.
//
// velog.io SparseVILA summary §3.2 (why decode-time selection is efficient):
// the selected KV entries are gathered into contiguous memory so that the
// decode attention reads them with regular, coalesced accesses instead of
// scattered rows.  Once per round, for every (sequence, KV head), the K/V
// rows of the retrieved visual tokens (in vis_idx order) and of all text
// tokens are copied to positions [0, k + n_text) of a second paged layer;
// dense attention over that layer then reads whole contiguous pages.
//
// HBM-bound copy: each thread moves 16-byte pieces; a CTA covers 32 tokens
// of one (KV head, sequence), K then V.
#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {
constexpr int kPackTokens = 32;
constexpr int kPackThreads = 256;
}  // namespace

__global__ void __launch_bounds__(kPackThreads)
pack_kv_kernel(const uint4* __restrict__ k_src, const uint4* __restrict__ v_src, int src_blocks,
               const int32_t* __restrict__ src_bt, int src_max_blocks, int n_vis,
               const int32_t* __restrict__ vis_idx, int k, int n_text, uint4* __restrict__ k_dst,
               uint4* __restrict__ v_dst, int dst_blocks, const int32_t* __restrict__ dst_bt,
               int dst_max_blocks, int Hkv, int vecs_per_tok, int* status) {
  grid_dep_sync();
  const int g = blockIdx.y, b = blockIdx.z;
  const int t0 = blockIdx.x * kPackTokens;
  const int n_tok = k + n_text;
  const int ntile = min(kPackTokens, n_tok - t0);
  const int32_t* sbt = src_bt + (size_t)b * src_max_blocks;
  const int32_t* dbt = dst_bt + (size_t)b * dst_max_blocks;
  const int32_t* vrow = vis_idx ? vis_idx + ((size_t)b * Hkv + g) * k : nullptr;
  const int pieces = ntile * vecs_per_tok;
  for (int p = threadIdx.x; p < pieces; p += kPackThreads) {
    const int t = t0 + p / vecs_per_tok, v = p % vecs_per_tok;
    int pos;
    if (t < k) {
      pos = vrow ? __ldg(vrow + t) : t;
      if (pos < 0 || pos >= n_vis) {
        if (v == 0) flag_status(status, kStatusBadIndex);
        continue;
      }
    } else {
      pos = n_vis + (t - k);
    }
    const int spage = __ldg(sbt + (pos >> 4)), dpage = __ldg(dbt + (t >> 4));
    if (spage < 0 || spage >= src_blocks || dpage < 0 || dpage >= dst_blocks) {
      if (v == 0) flag_status(status, kStatusBadBlock);
      continue;
    }
    const long long so = ((((long long)spage * Hkv + g) << 4) + (pos & 15)) * vecs_per_tok + v;
    const long long dof = ((((long long)dpage * Hkv + g) << 4) + (t & 15)) * vecs_per_tok + v;
    const uint4 kv = ld_stream16(k_src + so);
    const uint4 vv = ld_stream16(v_src + so);
    k_dst[dof] = kv;
    v_dst[dof] = vv;
  }
}

cudaError_t launch_pack_kv(const void* k_src, const void* v_src, int src_blocks, const int32_t* src_bt,
                           int src_max_blocks, int n_vis, const int32_t* vis_idx, int k, int n_text,
                           void* k_dst, void* v_dst, int dst_blocks, const int32_t* dst_bt,
                           int dst_max_blocks, int batch, int Hkv, int D, int* status,
                           cudaStream_t stream) {
  const int n_tok = k + n_text;
  if (batch == 0 || n_tok == 0) return cudaSuccess;
  dim3 grid((n_tok + kPackTokens - 1) / kPackTokens, Hkv, batch);
  return launch_dependent(pack_kv_kernel, grid, dim3(kPackThreads), 0, stream, static_cast<const uint4*>(k_src),
                          static_cast<const uint4*>(v_src), src_blocks, src_bt, src_max_blocks, n_vis, vis_idx, k,
                          n_text, static_cast<uint4*>(k_dst), static_cast<uint4*>(v_dst), dst_blocks, dst_bt,
                          dst_max_blocks, Hkv, D / 8, status);
}

}  // namespace sv
