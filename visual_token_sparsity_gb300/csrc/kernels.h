// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace sv {

// Optional per-sequence lengths of a decode batch: device int32 arrays of
// `batch` entries, nullptr = the batch-wide value for every sequence.  With
// any of them set, the batch-wide n_vis / n_text / k are capacities: strides
// of the score and index arrays, workspace sizes and split plans.
struct SeqLens {
  const int32_t* n_vis = nullptr;   // visual tokens of each sequence
  const int32_t* n_text = nullptr;  // text tokens of each sequence
  const int32_t* k = nullptr;       // selected visual tokens of each sequence
  __host__ __device__ bool any() const { return n_vis || n_text || k; }
};

// ---- retrieval scoring + top-k (retrieve.cu).  With row_done (zeroed int per
// (sequence, KV head) row) and rows that fit in shared memory, the top-k runs
// inside the scoring kernel; otherwise a separate top-k kernel follows.
// Per-sequence lengths: scores of sequence b cover its n_vis[b] tokens, its
// rows select k[b] indices and fill the rest of the k slots with -1.
cudaError_t launch_retrieve(const void* q, int R, int H, int G, const void* k_pool, int num_blocks,
                            int Hkv, int D, const int32_t* block_table, int max_blocks, int n_vis,
                            int batch, float* scores, int* status, int num_sms, int* row_done, int k,
                            int32_t* vis_idx, cudaStream_t stream, const SeqLens& lens = SeqLens{},
                            int n_text = 0);

// ---- softmax-normalised retrieval (retrieve_softmax.cu): scores of visual
// tokens = attention mass of the R x G question rows, then the row top-k
size_t retrieve_softmax_workspace_bytes(int B, int R, int H, int Hkv, int D, int n_vis, int n_text);
int retrieve_softmax_max_rows();
cudaError_t launch_retrieve_softmax(const void* q, int R, int H, float scale, const void* k_pool, int num_blocks,
                                    int Hkv, int D, const int32_t* block_table, int max_blocks, int n_vis,
                                    int n_text, int batch, const float* lse_in, int k, int32_t* vis_idx,
                                    float* scores_out, void* ws, int* status, cudaStream_t stream);

// ---- row top-k (topk.cu: one CTA per row; topk_cluster.cu: an 8-CTA cluster
// per row for long rows).  n and k are the row stride of scores and idx; with
// per-sequence lengths (rows_per_seq rows per sequence) row r uses
// lens.n_vis / lens.k of sequence r / rows_per_seq and fills its slots past
// that k with -1 (out-of-range lengths: the whole row is -1).
cudaError_t launch_topk_rows(const float* scores, int rows, int n, int k, int32_t* idx,
                             cudaStream_t stream, const SeqLens& lens = SeqLens{}, int rows_per_seq = 1);
bool topk_cluster_fits(int n);
bool topk_prefers_cluster(int n);   // long rows that fit: use launch_topk_cluster
cudaError_t launch_topk_cluster(const float* scores, int rows, int n, int k, int32_t* idx,
                                cudaStream_t stream, const SeqLens& lens = SeqLens{},
                                int rows_per_seq = 1);

// ---- pack-once KV (pack.cu): selected visual + text rows of src copied to
// positions [0, k + n_text) of every sequence of dst (same Hkv and D)
cudaError_t launch_pack_kv(const void* k_src, const void* v_src, int src_blocks, const int32_t* src_bt,
                           int src_max_blocks, int n_vis, const int32_t* vis_idx, int k, int n_text,
                           void* k_dst, void* v_dst, int dst_blocks, const int32_t* dst_bt,
                           int dst_max_blocks, int batch, int Hkv, int D, int* status,
                           cudaStream_t stream);

// ---- sparse decode attention (attn.cu)
struct AttnPlan {
  int tile;
  int chunk;   // tokens per split (multiple of tile)
  int nsplit;  // splits per (sequence, KV head)
  int nsplit_max;  // upper bound of nsplit over all n' <= n_tokens
};
AttnPlan attn_plan(int B, int Hkv, int G, int n_tokens);
// kernels one attention call launches: 1 (split merge fused), or 2 (merge kernel)
int attn_kernel_count(int B, int Hkv, int G, int n_tokens);
// whether the retrieval top-k runs inside the scoring kernel (rows of n_vis keys)
bool retrieve_fuses_topk(int rows, int n_vis);

struct AttnArgs {
  const void* q;
  int H;
  float scale;
  const void* k_pool;
  const void* v_pool;
  int num_blocks, Hkv, D;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* vis_idx;
  int k_vis, n_vis, n_text, batch;   // capacities when lens has per-sequence counts
  SeqLens lens;                       // vis_idx == nullptr: lens.k is ignored (all visual tokens)
  void* out;
  float* lse;
  float* part_ml;
  float* part_o;
  int* split_done;   // zeroed int per (sequence, KV head); left zeroed after the call
  int* status;
  // fused append: one new token per (sequence, KV head), bf16 [batch][Hkv][D],
  // stored at text position n_text and attended as the last token (n_text
  // then counts the tokens before it); nullptr: plain attention
  const void* k_new = nullptr;
  const void* v_new = nullptr;
};
cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream);
cudaError_t launch_sparse_attn_mma(const AttnArgs& a, const AttnPlan& p, cudaStream_t stream);

// ---- compaction gather (prune.cu)
cudaError_t launch_gather_rows(const void* feat, int B, int N, int k, int64_t row_bytes,
                               const int32_t* idx, void* out, int* status, cudaStream_t stream,
                               const int32_t* counts = nullptr);
cudaError_t launch_threshold_select(const float* sal, int B, int N, float threshold, int32_t* idx, int32_t* count,
                                    cudaStream_t stream);

// ---- cache maintenance (evict.cu)
cudaError_t launch_kv_move_down(void* k_pool, void* v_pool, int num_blocks, int Hkv, int D,
                                const int32_t* block_table, int max_blocks, int batch,
                                int dst_pos, int src_pos, int count, int* status,
                                cudaStream_t stream);
// new tokens go to positions [pos0, pos0 + T); with per-sequence lengths
// pos0 of sequence b is lens.n_vis[b] + lens.n_text[b] (each falling back to
// n_vis / n_text), and pos0 is unused
cudaError_t launch_kv_append(void* k_pool, void* v_pool, int num_blocks, int Hkv, int D,
                             const int32_t* block_table, int max_blocks, int batch, int pos0,
                             const void* k_new, const void* v_new, int T, int* status,
                             cudaStream_t stream, const SeqLens& lens = SeqLens{}, int n_vis = 0,
                             int n_text = 0);

// ---- prefill salience (salience.cu)
cudaError_t launch_head_mean(const float* colsum, int B, int H, int N, float inv, float* out,
                             cudaStream_t stream);
// ---- summary-row salience (summary.cu)
size_t summary_smem_bytes(int N, int d, int R);
cudaError_t launch_summary_salience(const void* q, const void* k, int B, int H, int N, int d, int R,
                                    float scale, float* salience, float* colsum, cudaStream_t stream);
bool salience_head_dim_supported(int d);
// whether sv_salience_prefill streams both operands (long sequences) and how
// many kernels one call launches
bool salience_uses_long_schedule(int N, int d);
int salience_kernel_count(int N, int d);
size_t salience_workspace_bytes(int B, int H, int N, int d);
cudaError_t launch_salience(const void* q, const void* k, int B, int H, int N, int d, float scale,
                            float* salience, void* ws, int* status, int num_sms,
                            cudaStream_t stream);

}  // namespace sv
