// Paged-cache maintenance between conversation rounds.
//
// velog.io SparseVILA summary §4.1 Setup: after each round only the previous
// question/answer KV entries are evicted and the visual cache is kept
// (xllm-io review §五 partial_kv_cache_eviction).  A span that ends at the
// tail is removed by shortening the text length on the host; a span in the
// middle is removed by moving the later text tokens down, which this kernel
// does in place.
#include "common.cuh"
#include "kernels.h"

namespace sv {

namespace {

__device__ __forceinline__ long long token_vec(const int32_t* bt, int num_blocks, int Hkv, int g,
                                               int pos, int vecs_per_tok, int* status) {
  const int page = __ldg(bt + (pos >> 4));
  if (page < 0 || page >= num_blocks) {
    flag_status(status, kStatusBadBlock);
    return -1;
  }
  return ((((long long)page * Hkv + g) << 4) + (pos & 15)) * vecs_per_tok;
}

}  // namespace

// One CTA per (KV head, sequence).  Tokens move in chunks no longer than the
// shift, so a chunk's destination never overlaps a source that is still to
// be read; each chunk is loaded completely before any of it is stored.
__global__ void __launch_bounds__(256)
kv_move_down_kernel(uint4* k_pool, uint4* v_pool, int num_blocks, int Hkv, int vecs_per_tok,
                    const int32_t* __restrict__ block_table, int max_blocks, int dst_pos,
                    int src_pos, int count, int* status) {
  grid_dep_sync();
  const int g = blockIdx.x, b = blockIdx.y;
  const int32_t* bt = block_table + (size_t)b * max_blocks;
  const int shift = src_pos - dst_pos;
  const int chunk = shift < 32 ? shift : 32;
  for (int done = 0; done < count; done += chunk) {
    const int n = min(chunk, count - done);
    const int total = n * vecs_per_tok * 2;
    uint4 buf[8];
    long long dst_off[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int piece = threadIdx.x + 256 * i;
      dst_off[i] = -1;
      if (piece < total) {
        const int tensor = piece / (n * vecs_per_tok);
        const int rem = piece % (n * vecs_per_tok);
        const int t = rem / vecs_per_tok, v = rem % vecs_per_tok;
        const long long so = token_vec(bt, num_blocks, Hkv, g, src_pos + done + t, vecs_per_tok, status);
        const long long doff = token_vec(bt, num_blocks, Hkv, g, dst_pos + done + t, vecs_per_tok, status);
        if (so >= 0 && doff >= 0) {
          buf[i] = (tensor ? v_pool : k_pool)[so + v];
          dst_off[i] = (doff + v) | ((long long)tensor << 62);
        }
      }
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (dst_off[i] >= 0) {
        const bool is_v = (dst_off[i] >> 62) & 1;
        const long long off = dst_off[i] & ((1LL << 62) - 1);
        (is_v ? v_pool : k_pool)[off] = buf[i];
      }
    }
    __syncthreads();
  }
}

cudaError_t launch_kv_move_down(void* k_pool, void* v_pool, int num_blocks, int Hkv, int D,
                                const int32_t* block_table, int max_blocks, int batch,
                                int dst_pos, int src_pos, int count, int* status,
                                cudaStream_t stream) {
  if (count <= 0 || batch == 0) return cudaSuccess;
  dim3 grid(Hkv, batch);
  return launch_dependent(kv_move_down_kernel, grid, dim3(256), 0, stream, static_cast<uint4*>(k_pool),
                          static_cast<uint4*>(v_pool), num_blocks, Hkv, D / 8, block_table, max_blocks, dst_pos,
                          src_pos, count, status);
}

// Writes new tokens' K/V rows ([B][T][Hkv][d], token-major) into their pages,
// at [pos0, pos0 + T) or, with per-sequence lengths, after each sequence's
// own visual and text tokens (capacities n_vis, n_text keep every position
// inside the block table).
__global__ void __launch_bounds__(256)
kv_append_kernel(uint4* k_pool, uint4* v_pool, int num_blocks, int Hkv, int vecs_per_tok,
                 const int32_t* __restrict__ block_table, int max_blocks, int pos0,
                 const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, int T,
                 long long total, int* status, SeqLens lens, int n_vis, int n_text) {
  grid_dep_sync();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int v = (int)(i % vecs_per_tok);
    long long r = i / vecs_per_tok;
    const int g = (int)(r % Hkv);
    r /= Hkv;
    const int t = (int)(r % T);
    const int b = (int)(r / T);
    int p0 = pos0;
    if (lens.any()) {
      SeqLens l = lens;
      l.k = nullptr;
      int nv, nt, kb;
      if (!seq_lengths(l, b, n_vis, n_text, 0, nv, nt, kb)) {
        if (v == 0 && g == 0 && t == 0) flag_status(status, kStatusBadLength);
        continue;
      }
      p0 = nv + nt;
    }
    const long long off = token_vec(block_table + (size_t)b * max_blocks, num_blocks, Hkv, g,
                                    p0 + t, vecs_per_tok, status);
    if (off < 0) continue;
    k_pool[off + v] = k_new[i];
    v_pool[off + v] = v_new[i];
  }
}

cudaError_t launch_kv_append(void* k_pool, void* v_pool, int num_blocks, int Hkv, int D,
                             const int32_t* block_table, int max_blocks, int batch, int pos0,
                             const void* k_new, const void* v_new, int T, int* status,
                             cudaStream_t stream, const SeqLens& lens, int n_vis, int n_text) {
  const long long total = (long long)batch * T * Hkv * (D / 8);
  if (total == 0) return cudaSuccess;
  long long blocks = (total + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  return launch_dependent(kv_append_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                          static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), num_blocks, Hkv, D / 8,
                          block_table, max_blocks, pos0, static_cast<const uint4*>(k_new),
                          static_cast<const uint4*>(v_new), T, total, status, lens, n_vis, n_text);
}

}  // namespace sv
