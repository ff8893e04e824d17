/*
 * sv.h -- C ABI of libsv, the GB300 (sm_103a) SparseVILA hot path.
 *
 * The operations follow "SparseVILA: Decoupling Visual Sparsity for Efficient
 * VLM Inference" (arXiv 2510.17777) as summarised on velog.io (§2 table, §3.1
 * Prefill Phase, §3.2 Decode Phase, §4.1 Setup) and reviewed on xllm-io
 * (§三 core formulas, §五 code analysis):
 *   prefill  -- query-agnostic salience from the encoder's self-attention,
 *               top-k prune and compaction of the kept tokens;
 *   decode   -- query-aware retrieval of the most relevant cached visual
 *               tokens and attention over them plus all text tokens;
 *   rounds   -- partial eviction of the previous question/answer KV.
 *
 * General conventions (every call):
 *   - All tensor pointers are DEVICE pointers owned by the caller unless the
 *     comment says "host".  The library allocates no memory of its own; each
 *     call (except sv_retrieve_topk_noalloc) takes a caller-owned device
 *     workspace `ws` of at least the size the matching
 *     sv_*_workspace_bytes() returns.  The first 256 bytes of every
 *     workspace hold the device status word (see sv_read_device_status); a
 *     fresh workspace must be zero-filled once before first use.  Calls that
 *     share a workspace must be ordered on one stream.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously; nothing synchronises except
 *     sv_read_device_status and, for non-tail spans, nothing in
 *     sv_evict_qa_tokens either.  No call allocates, frees or synchronises;
 *     the workspace-taking compute calls may be captured in a CUDA graph.
 *   - The return value covers host-side argument checks and the launch
 *     (cudaGetLastError).  On an error nothing is launched and
 *     sv_last_error() returns a description (thread-local).
 *   - Device-side index errors (a block id outside the pool, a visual index
 *     outside [0, n_vis), a per-sequence length outside its capacity) set a
 *     bit in the status word; the offending load (or sequence) is skipped.
 *     Kernels never trap.
 *   - bf16 tensors are IEEE bfloat16 bit patterns (uint16).  Accumulation is
 *     fp32.  No C++ exception crosses this ABI.
 *   - GQA: query head h reads KV head h / G with G = H / Hkv.
 */
#ifndef SV_H_
#define SV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,   /* a null pointer, a size out of range, k > n ... */
  SV_ERR_UNSUPPORTED = 2,   /* a head_dim or shape the library has no kernel for */
  SV_ERR_CUDA = 3,          /* a CUDA runtime error while launching */
  SV_ERR_WORKSPACE = 4,     /* ws_bytes smaller than required */
  SV_ERR_DEVICE_BOUNDS = 5  /* reported by sv_read_device_status only */
} sv_status;

/* Device status bits (the status word is the first int32 of a workspace). */
#define SV_DEV_BAD_BLOCK 0x1   /* a block-table entry outside [0, num_blocks) */
#define SV_DEV_BAD_INDEX 0x2   /* a visual index outside [0, n_vis) */
#define SV_DEV_BAD_LENGTH 0x4  /* a per-sequence length outside its capacity; that sequence is skipped */
#define SV_DEV_TIMEOUT   0x10  /* a bounded wait inside a kernel gave up (2 s); results undefined */

/* Tokens per KV page (fixed). */
#define SV_BLOCK_TOKENS 16

const char* sv_status_string(sv_status s);
/* Thread-local description of the last error returned on this thread. */
const char* sv_last_error(void);
/* Library version string, e.g. "sv 0.1 sm_103a". */
const char* sv_version(void);

/*
 * One layer's paged KV cache (caller-owned device memory).
 * k_pool, v_pool: bf16 [num_blocks][n_kv_heads][16][head_dim].  Each page
 * holds 16 consecutive logical positions of one sequence for every KV head.
 */
typedef struct {
  void* k_pool;
  void* v_pool;
  int32_t num_blocks;
  int32_t n_kv_heads;
  int32_t head_dim;
} sv_kv_layer;

/*
 * A batch of sequences sharing one block table (same table for every layer).
 * block_table: DEVICE int32 [batch][max_blocks]; logical position t of
 * sequence b lives in page block_table[b][t / 16], row t % 16.
 * Logical layout of every sequence: visual tokens at [0, n_vis), then n_text
 * text tokens.
 *
 * Per-sequence lengths (xllm-io review §五: a threshold prune keeps a
 * different number of visual tokens per frame or sequence).  The three
 * optional DEVICE int32 [batch] arrays below give each sequence its own
 * counts; NULL means the batch-wide value.  With any of them set, n_vis,
 * n_text and the calls' k are CAPACITIES: every per-sequence count must lie
 * in [0, capacity] (and k_seq[b] <= n_vis_seq[b]); score rows keep the stride
 * n_vis, index rows the stride k, split plans and workspaces are sized for
 * the capacities.  Sequence b's visual tokens sit at [0, n_vis_seq[b]) and
 * its text right after them, at [n_vis_seq[b], n_vis_seq[b] + n_text_seq[b]).
 * A sequence whose counts are out of range sets SV_DEV_BAD_LENGTH and is
 * skipped (its indices read -1, its attention output 0).
 * Accepted by sv_retrieve_topk, sv_retrieve_topk_noalloc,
 * sv_sparse_decode_attn and sv_kv_append; the other calls taking a batch
 * return SV_ERR_UNSUPPORTED when any of the arrays is set.
 * Zero-initialise the struct so that the arrays default to NULL.
 */
typedef struct {
  const int32_t* block_table;
  int32_t batch;
  int32_t max_blocks;
  int32_t n_vis;
  int32_t n_text;
  const int32_t* n_vis_seq;   /* optional [batch]: visual tokens of each sequence */
  const int32_t* n_text_seq;  /* optional [batch]: text tokens of each sequence */
  const int32_t* k_seq;       /* optional [batch]: selected visual tokens of each sequence */
} sv_seq_batch;

/* ------------------------------------------------------------------------
 * Workspace sizes (bytes, always >= 256).  Pure host functions.
 */
size_t sv_salience_workspace_bytes(int B, int H, int N, int d);
size_t sv_topk_workspace_bytes(int rows, int n, int k);
size_t sv_prune_workspace_bytes(int B, int N, int k);
size_t sv_retrieve_workspace_bytes(int B, int H, int n_kv_heads, int head_dim, int n_vis, int k);
size_t sv_attn_workspace_bytes(int B, int H, int n_kv_heads, int head_dim, int n_tokens);
size_t sv_evict_workspace_bytes(void);

/*
 * Kernels one call launches on its stream (pure host functions, for callers
 * that budget launches, e.g. when building CUDA graphs):
 *   sv_retrieve_kernel_count -- sv_retrieve_topk over batch * n_kv_heads
 *     rows of n_vis keys: 1 (the top-k runs inside the scoring kernel: at
 *     most 64 rows of at most 11264 keys) or 2 (a separate top-k kernel);
 *     0 for n_vis <= 0.
 *   sv_attn_kernel_count -- sv_sparse_decode_attn over n_tokens attended
 *     tokens per (sequence, KV head): 1 (the split merge runs inside the
 *     attention kernel) or 2 (a separate merge kernel); 0 for invalid sizes.
 */
int sv_retrieve_kernel_count(int batch, int n_kv_heads, int n_vis);
/* sv_salience_prefill over N tokens of head dim d: 3 (salience kernel, its
 * exact re-run of failed heads, head mean) or 4 for long sequences (row
 * pass, its re-run, column pass, head mean); 0 for unsupported sizes. */
int sv_salience_kernel_count(int N, int d);
int sv_attn_kernel_count(int B, int H, int n_kv_heads, int n_tokens);

/* ------------------------------------------------------------------------
 * Prefill salience -- velog.io summary §3.1 (salience table, "no summary
 * token" encoders such as SigLIP / QwenVL: the intra-visual attention a token
 * receives, averaged over all tokens; kernel paragraph: softmax normalisation
 * and salience accumulation streamed without materialising the attention
 * matrix); xllm-io review §三 salience formula.
 *
 *   salience[b][j] = 1/(H*N) * sum_h sum_i softmax_j(scale * q[b,h,i,:] . k[b,h,j,:])
 *
 * q, k     : bf16 [B][H][N][d], contiguous.
 * scale    : logit scale (1/sqrt(d) for standard attention); must be > 0.
 * salience : out fp32 [B][N]; each row sums to 1.
 * Supported: d in {64, 72, 80, 128}, 1 <= N <= 2^24; other head dims return
 * SV_ERR_UNSUPPORTED.  Computed with tcgen05 tensor-core tiles (bf16
 * operands, fp32 accumulation) in two passes -- row log-sum-exp, then column
 * accumulation with -lse folded into the MMA -- without forming the N x N
 * matrix.  Short sequences (N <= 1024 at d 64 / 72, 768 at d 80, 512 at
 * d 128) keep one head's keys or queries resident in shared memory; longer
 * ones stream both operands through 128 x 256 tiles.  Row sums are taken without a running
 * max; heads whose sums leave [2^-90, 2^100] are recomputed with one by a
 * second, normally empty, launch.  Deterministic.
 * ws_bytes >= sv_salience_workspace_bytes(B, H, N, d).
 */
sv_status sv_salience_prefill(const void* q, const void* k, int B, int H, int N, int d,
                              float scale, float* salience, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * Query-agnostic salience for encoders with summary tokens -- velog.io
 * summary §3.1 encoder-type table: one summary token (CLIP), a token's
 * importance is the attention it contributes to the summary token; several
 * (RADIO), the mean attention toward them.  The R summary tokens are the
 * first R tokens of the sequence:
 *
 *   salience[b][j] = 1/(H*R) * sum_h sum_{r<R} softmax_j(scale * q[b,h,r,:] . k[b,h,j,:])
 *
 * (softmax over all N tokens; summary columns are reported too).
 * q, k     : bf16 [B][H][N][d], contiguous (only rows r < R of q are read).
 * R        : 1 <= R <= min(16, N); R * N logits per head must fit in shared
 *            memory (R * N <= ~56K).  d: a multiple of 8, at most 256.
 * salience : out fp32 [B][N]; each row sums to 1.
 * Only R rows of each head's attention map are formed: one CTA per (frame,
 * head) streams K once (HBM-bound), then a head-mean kernel.  Deterministic.
 */
size_t sv_salience_summary_workspace_bytes(int B, int H, int N, int d, int R);
sv_status sv_salience_summary(const void* q, const void* k, int B, int H, int N, int d, int R,
                              float scale, float* salience, void* ws, size_t ws_bytes, void* stream);

/*
 * Row-wise top-k (the selection step shared by prefill pruning and decode
 * retrieval) -- velog.io summary §3.1 (drop the lowest-salience tokens) and
 * §3.2 (activate the highest-scoring tokens); xllm-io review §五 topk.
 *
 * scores : fp32 [rows][n].
 * idx    : out int32 [rows][k]: the k largest entries of each row, ties broken
 *          towards the lower index (-0.0 equals +0.0), written in ascending
 *          index order.  NaN scores give an unspecified (but valid) choice.
 * 1 <= k <= n <= 2^24.
 */
sv_status sv_topk_rows(const float* scores, int rows, int n, int k, int32_t* idx, void* ws,
                       size_t ws_bytes, void* stream);

/*
 * Prefill prune + compaction -- velog.io summary §2 table (prefill tokens are
 * actually deleted) and §3.1; xllm-io review §五 query_agnostic_pruning.
 *
 * salience  : fp32 [B][N] (e.g. from sv_salience_prefill).
 * feat      : [B][N][row_bytes] opaque rows (row_bytes % 16 == 0, base 16-byte aligned).
 * feat_out  : out [B][k][row_bytes]: the kept rows in ascending token order.
 * kept_idx  : out int32 [B][k] ascending.
 */
sv_status sv_prune_compact(const float* salience, int B, int N, int k, const void* feat,
                           int64_t row_bytes, void* feat_out, int32_t* kept_idx, void* ws,
                           size_t ws_bytes, void* stream);

/*
 * Prefill prune by a salience threshold -- xllm-io review §五
 * query_agnostic_pruning (keep the tokens whose salience exceeds the
 * threshold): a variable number of tokens per frame.
 *
 * salience   : fp32 [B][N]; a token is kept iff salience > threshold
 *              (strictly; NaN scores are dropped; a NaN threshold is an error).
 * feat       : [B][N][row_bytes] opaque rows (row_bytes a multiple of 16; 0 = no rows).
 * feat_out   : out [B][N][row_bytes]: rows [0, kept_count[b]) of frame b hold
 *              the kept rows in token order; later rows are not written.
 * kept_idx   : out int32 [B][N]: the kept indices ascending, then -1.
 * kept_count : out device int32 [B].
 * ws         : sv_prune_workspace_bytes(B, N, 1) (the status word).
 */
sv_status sv_prune_threshold(const float* salience, int B, int N, float threshold, const void* feat,
                             int64_t row_bytes, void* feat_out, int32_t* kept_idx, int32_t* kept_count,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * Decode query-aware retrieval -- velog.io summary §3.2 "Query-Aware Token
 * Selection" (text query as Query, cached visual tokens as Keys, aggregate
 * attention strength; the rest stays cached but inactive); xllm-io review §三
 * Selected = TopK(Query . KV_Cache, k) and §五 query_aware_retrieval.
 *
 *   score[b][g][j] = sum_{r<R} sum_{h in group g} q[b,r,h,:] . K[b,g,j,:],  j < n_vis
 *   vis_idx[b][g]  = top-k of score[b][g]  (ties -> lower index, ascending)
 *
 * q        : bf16 [B][R][H][d] (the current question's query rows).
 * layer    : the layer's paged cache; seqs: batch view (n_vis, or the
 *            per-sequence n_vis_seq and k_seq).
 * vis_idx  : out int32 [B][Hkv][k].  With k_seq, row (b, g) holds k_seq[b]
 *            ascending indices and -1 in its remaining slots.
 * scores   : optional out fp32 [B][Hkv][n_vis] (NULL = not written; with
 *            n_vis_seq only the first n_vis_seq[b] entries of a row).
 * Supported: d in {64, 128}; 1 <= k <= n_vis; H % Hkv == 0.
 */
sv_status sv_retrieve_topk(const void* q, int R, int H, const sv_kv_layer* layer,
                           const sv_seq_batch* seqs, int k, int32_t* vis_idx, float* scores,
                           void* ws, size_t ws_bytes, void* stream);

/*
 * sv_retrieve_topk without a workspace.  (No counterpart on the SparseVILA
 * pages: this is a calling convenience, not part of the method.)
 *
 * Some callers cannot allocate device memory at all -- for example a plugin
 * running inside a host framework that owns all device memory through its
 * own pool, or a latency-critical loop where cudaMalloc (which can
 * synchronise the device) is forbidden -- so they cannot supply the scores
 * workspace sv_retrieve_topk needs.  This entry point computes exactly what
 * sv_retrieve_topk computes (the same scoring kernel and the same top-k
 * routine, here always run as a separate top-k kernel), keeping the scores in
 * a fixed scratch array compiled into the library (8 MiB + 256 B of device
 * memory on every GPU that loads the library, held until the process exits).
 *
 * Arguments are those of sv_retrieve_topk minus ws / ws_bytes.  It allocates
 * nothing and calls no allocating routine.
 * Limit: batch * n_kv_heads * n_vis <= 2^21 (2,097,152 scores); larger calls
 * return SV_ERR_WORKSPACE without launching.
 * Every call looks up the scratch array's device address
 * (cudaGetSymbolAddress) on the current device.  With lazy module loading
 * (the CUDA default) the first call on each device loads this code and maps
 * the 8 MiB array at that moment, which can fail with SV_ERR_CUDA (out of
 * memory) when the caller's pool already holds nearly all device memory:
 * make that first call at start-up, before any stream capture.
 * All calls share the one scratch array: calls that can overlap on the GPU
 * (different streams without ordering, or several host threads) race and
 * must not be issued.  The status word at the start of the scratch is
 * cleared by every call; device-side index errors are skipped as in
 * sv_retrieve_topk but cannot be read back through sv_read_device_status.
 */
sv_status sv_retrieve_topk_noalloc(const void* q, int R, int H, const sv_kv_layer* layer,
                                   const sv_seq_batch* seqs, int k, int32_t* vis_idx, float* scores,
                                   void* stream);

/*
 * Softmax-normalised query-aware retrieval -- velog.io summary §3.2
 * ("aggregated attention strength" between the question's rows and the
 * cached vision tokens; the pages' retrieval runs alongside the question's
 * FlashAttention-2 prefill).  Per sequence b and KV head g:
 *
 *   score[b][g][j] = sum_{r<R} sum_{h in g} exp(scale * q[b,r,h] . K[b,g,j] - lse[b,r,h]),  j < n_vis
 *   vis_idx[b][g]  = the k largest scores, ascending (ties -> lower index)
 *
 * lse : optional fp32 [B][R][H], natural log: each question row's softmax
 *       normaliser from the caller's own prefill attention (the fused form;
 *       no extra pass).  NULL: computed here over all n_vis + n_text cached
 *       tokens, no causal mask (one extra pass over K).
 * q   : bf16 [B][R][H][d]; R * (H / n_kv_heads) <= 256; d in {64, 128}.
 * scores (optional out fp32 [B][Hkv][n_vis]), vis_idx, ws as sv_retrieve_topk;
 * ws_bytes >= sv_retrieve_softmax_workspace_bytes(...).
 * The logits are warp-level tensor-core tiles over the question rows of
 * each KV head; deterministic.
 */
size_t sv_retrieve_softmax_workspace_bytes(int B, int R, int H, int n_kv_heads, int head_dim, int n_vis,
                                           int n_text);
sv_status sv_retrieve_topk_softmax(const void* q, int R, int H, float scale, const sv_kv_layer* layer,
                                   const sv_seq_batch* seqs, const float* lse, int k, int32_t* vis_idx,
                                   float* scores, void* ws, size_t ws_bytes, void* stream);

/*
 * Sparse decode attention -- velog.io summary §3.2 (only the query-relevant
 * subset of the preserved visual cache is read) and §4.5 kernel table
 * ("decoding attention": reduced KV, less memory traffic).
 *
 *   T[b][g] = vis_idx[b][g][0..k) U [n_vis, n_vis + n_text)
 *   out[b][h] = sum_{t in T} softmax_t(scale * q[b,h] . K[b,g,t]) V[b,g,t],  g = h / G
 *
 * q       : bf16 [B][H][d] (one decode query per head).
 * vis_idx : int32 [B][Hkv][k], distinct values in [0, n_vis); NULL = all
 *           n_vis visual tokens (dense attention; k is then ignored).
 *           Per-sequence lengths: sequence b attends to the first k_seq[b]
 *           entries of its rows (values in [0, n_vis_seq[b])) and to its
 *           n_text_seq[b] text tokens at [n_vis_seq[b], + n_text_seq[b]);
 *           with vis_idx NULL, to all its n_vis_seq[b] visual tokens.
 * out     : out bf16 [B][H][d].
 * lse     : optional out fp32 [B][H], log sum_t exp(scale q.k_t) (NULL = none).
 * Split-K over tokens with an fp32 online softmax; per-split partials live in
 * ws and are merged in the same kernel (or a second one when there are many
 * splits).  G <= 2 uses CUDA-core dot products, 3 <= G <= 16 warp-level
 * tensor-core tiles.  Supported: d in {64, 128}, G = H / Hkv <= 16.
 */
sv_status sv_sparse_decode_attn(const void* q, int H, float scale, const sv_kv_layer* layer,
                                const sv_seq_batch* seqs, const int32_t* vis_idx, int k,
                                void* out, float* lse, void* ws, size_t ws_bytes, void* stream);

/*
 * Pack-once KV for round reuse -- velog.io summary §3.2 (why decode-time
 * selection is efficient: the selected KV entries are gathered into
 * contiguous memory so the attention reads them with coalesced accesses).
 *
 * For every sequence b and KV head g, copies the K/V rows of the selected
 * visual tokens vis_idx[b][g][0..k) (in that order; NULL = all n_vis visual
 * tokens, k ignored) followed by the seqs->n_text text tokens of `src` to
 * logical positions [0, k + n_text) of sequence b in `dst`, addressed
 * through dst_seqs->block_table.  Afterwards
 *   sv_sparse_decode_attn(q, H, scale, dst, dst_seqs, NULL, 0, ...)
 * attends over the same tokens, in the same order and with the same split
 * plan, as sv_sparse_decode_attn(q, H, scale, src, seqs, vis_idx, k, ...),
 * and so returns the same bits, reading whole contiguous pages; later
 * decode tokens are appended to dst with sv_kv_append(dst, dst_seqs, ...).
 * src, seqs : the paged cache and its batch view (read only).
 * dst       : a second paged layer (own pools, same n_kv_heads / head_dim).
 * dst_seqs  : batch = seqs->batch, n_vis = k, n_text = seqs->n_text; its
 *             block table must cover k + n_text positions per sequence.
 * ws        : sv_evict_workspace_bytes() (the status word).
 * Device-side index / block errors set the status bits and skip the row.
 */
sv_status sv_pack_kv(const sv_kv_layer* src, const sv_seq_batch* seqs, const int32_t* vis_idx, int k,
                     const sv_kv_layer* dst, const sv_seq_batch* dst_seqs, void* ws, size_t ws_bytes,
                     void* stream);

/*
 * Partial KV-cache eviction between rounds -- velog.io summary §4.1 Setup
 * (after each round only the previous question/answer KV entries are removed;
 * the visual cache stays); xllm-io review §五 partial_kv_cache_eviction.
 *
 * Removes text-relative positions [text_begin, text_end) of every sequence
 * in every layer.  Visual pages are never touched.  A tail span
 * (text_end == n_text) only shortens seqs->n_text; otherwise the later text
 * tokens are moved down on the GPU (one kernel per layer on `stream`).
 * seqs           : host struct; n_text is updated on success.
 * n_blocks_in_use: optional host out int32 [batch]: pages each sequence still
 *                  needs (the caller owns free-page bookkeeping).
 */
sv_status sv_evict_qa_tokens(const sv_kv_layer* layers, int n_layers, sv_seq_batch* seqs,
                             int32_t text_begin, int32_t text_end, int32_t* n_blocks_in_use,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * Append T new tokens' K/V at logical positions [n_vis + n_text, + T) of every
 * sequence (a helper for driving rounds; the caller then adds T to n_text).
 * With per-sequence lengths: at [n_vis_seq[b] + n_text_seq[b], + T) of
 * sequence b (the caller then adds T to each n_text_seq entry); n_vis +
 * n_text + T must still fit in max_blocks * 16.
 * k_new, v_new: bf16 [B][T][Hkv][d].  The pages must already be in the table.
 */
sv_status sv_kv_append(const sv_kv_layer* layer, const sv_seq_batch* seqs, const void* k_new,
                       const void* v_new, int T, void* ws, size_t ws_bytes, void* stream);

/*
 * One decode step of a round in one launch: sv_kv_append(layer, seqs, k_new,
 * v_new, T = 1, ...) followed by sv_sparse_decode_attn over the selected
 * visual tokens and the n_text + 1 text tokens (the new token attends to
 * itself, as the last one).  Same results, bit for bit, as the two calls:
 * the new token's K and V are read from k_new / v_new and stored into the
 * cache at position n_vis + n_text (n_vis_seq[b] + n_text_seq[b] with
 * per-sequence lengths) for later steps; the caller then adds 1 to n_text,
 * as after sv_kv_append.  (No counterpart on the SparseVILA pages: the
 * velog.io summary §4.1 round protocol decodes its answer token by token;
 * fusing the append is a launch saving, not part of the method.)
 * q, vis_idx, k, out, lse: as for sv_sparse_decode_attn.
 * k_new, v_new: bf16 [B][Hkv][d], 16-byte aligned; n_vis + n_text + 1 must
 *               fit in max_blocks * 16, and the page must be in the table.
 * ws      : sv_attn_workspace_bytes(B, H, n_kv_heads, d, k + n_text + 1)
 *           (k = n_vis when vis_idx is NULL).
 * A block id outside the pool is reported (SV_DEV_BAD_BLOCK) and the new
 * token is then neither stored nor attended, as with the two calls.
 */
sv_status sv_decode_append_attn(const void* q, int H, float scale, const sv_kv_layer* layer,
                                const sv_seq_batch* seqs, const void* k_new, const void* v_new,
                                const int32_t* vis_idx, int k, void* out, float* lse, void* ws,
                                size_t ws_bytes, void* stream);

/*
 * Read (and optionally clear) the device status word of a workspace.
 * Synchronises `stream`.  status_out: host int32 (SV_DEV_* bits, 0 = clean).
 */
sv_status sv_read_device_status(void* ws, int clear, int32_t* status_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SV_H_ */
