// C-ABI entry points of libsv (declared in include/sv.h): argument checks,
// workspace layout and kernel launches.  No allocation, no synchronisation
// (except sv_read_device_status), no exceptions across the boundary.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "../../include/sv.h"
#include "api_checks.h"
#include "kernels.h"

namespace sv {

bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("SV_PDL");
    return !(e != nullptr && e[0] == '0');
  }();
  return on;
}
int topk_max_smem_keys();
}  // namespace sv

namespace {

constexpr size_t kStatusBytes = 256;
constexpr size_t kMaxSmemPerBlock = 232448;  // 227 KB opt-in on sm_100-family parts
thread_local char g_err[512] = "";

sv_status fail(sv_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

sv_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return SV_OK;
  return fail(SV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int num_sms() {
  int dev = 0, n = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int* status_word(void* ws) { return static_cast<int*>(ws); }

char* after_status(void* ws) { return static_cast<char*>(ws) + kStatusBytes; }

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

sv_status check_ws(void* ws, size_t have, size_t need) {
  if (!ws) return fail(SV_ERR_INVALID_ARG, "workspace pointer is NULL");
  if (!aligned16(ws)) return fail(SV_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (have < need) return fail(SV_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", have, need);
  return SV_OK;
}

// Per-sequence lengths of a batch view (all NULL: uniform lengths).
sv::SeqLens lens_of(const sv_seq_batch* S) {
  sv::SeqLens l;
  l.n_vis = S->n_vis_seq;
  l.n_text = S->n_text_seq;
  l.k = S->k_seq;
  return l;
}

sv_status reject_lens(const sv_seq_batch* S, const char* call) {
  if (S && lens_of(S).any())
    return fail(SV_ERR_UNSUPPORTED, "%s: per-sequence lengths (n_vis_seq / n_text_seq / k_seq) are not supported",
                call);
  return SV_OK;
}

}  // namespace

namespace sv {
// Records `msg` as this thread's sv_last_error() text.
void set_error_message(const char* msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

sv_status check_cache(const sv_kv_layer* L, const sv_seq_batch* S, bool need_v) {
  if (!L || !S) return fail(SV_ERR_INVALID_ARG, "layer or batch descriptor is NULL");
  if (!L->k_pool || (need_v && !L->v_pool) || !S->block_table)
    return fail(SV_ERR_INVALID_ARG, "cache pool or block table pointer is NULL");
  if (!aligned16(L->k_pool) || (need_v && !aligned16(L->v_pool)))
    return fail(SV_ERR_INVALID_ARG, "cache pools must be 16-byte aligned");
  if (L->head_dim != 64 && L->head_dim != 128)
    return fail(SV_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", L->head_dim);
  if (L->num_blocks <= 0 || L->n_kv_heads <= 0)
    return fail(SV_ERR_INVALID_ARG, "num_blocks and n_kv_heads must be positive");
  if ((long long)L->num_blocks * L->n_kv_heads * SV_BLOCK_TOKENS >= 0xffffffffLL)
    return fail(SV_ERR_UNSUPPORTED, "pool has too many rows for 32-bit row ids");
  if (S->batch < 0 || S->max_blocks <= 0 || S->n_vis < 0 || S->n_text < 0)
    return fail(SV_ERR_INVALID_ARG, "negative batch or length");
  if ((long long)S->n_vis + S->n_text > (long long)S->max_blocks * SV_BLOCK_TOKENS)
    return fail(SV_ERR_INVALID_ARG, "n_vis + n_text = %d exceeds max_blocks * 16 = %d",
                S->n_vis + S->n_text, S->max_blocks * SV_BLOCK_TOKENS);
  return SV_OK;
}

sv_status check_retrieve_args(const void* q, int R, int H, const sv_kv_layer* layer, const sv_seq_batch* seqs,
                              int k, const int32_t* vis_idx) {
  sv_status s = check_cache(layer, seqs, false);
  if (s != SV_OK) return s;
  if (!q || !vis_idx) return fail(SV_ERR_INVALID_ARG, "q and vis_idx must be non-NULL");
  if (!aligned16(q)) return fail(SV_ERR_INVALID_ARG, "q must be 16-byte aligned");
  const int Hkv = layer->n_kv_heads;
  if (R <= 0 || H <= 0 || H % Hkv) return fail(SV_ERR_INVALID_ARG, "need R > 0 and H a multiple of n_kv_heads");
  if (seqs->n_vis <= 0) return fail(SV_ERR_INVALID_ARG, "no visual tokens to retrieve from");
  if (k < 1 || k > seqs->n_vis) return fail(SV_ERR_INVALID_ARG, "need 1 <= k <= n_vis (k = %d)", k);
  return SV_OK;
}
}  // namespace sv

using sv::check_cache;

extern "C" {

const char* sv_status_string(sv_status s) {
  switch (s) {
    case SV_OK: return "ok";
    case SV_ERR_INVALID_ARG: return "invalid argument";
    case SV_ERR_UNSUPPORTED: return "unsupported shape";
    case SV_ERR_CUDA: return "CUDA error";
    case SV_ERR_WORKSPACE: return "workspace too small";
    case SV_ERR_DEVICE_BOUNDS: return "device-side index out of bounds";
  }
  return "unknown status";
}

const char* sv_last_error(void) { return g_err; }

const char* sv_version(void) { return "sv 0.1 sm_103a"; }

// ------------------------------------------------------------------ sizes

size_t sv_salience_workspace_bytes(int B, int H, int N, int d) {
  if (B < 0 || H < 0 || N <= 0 || !sv::salience_head_dim_supported(d)) return kStatusBytes;
  return kStatusBytes + round256(sv::salience_workspace_bytes(B, H, N, d));
}

int sv_salience_kernel_count(int N, int d) {
  if (N <= 0 || !sv::salience_head_dim_supported(d)) return 0;
  return sv::salience_kernel_count(N, d);
}

size_t sv_topk_workspace_bytes(int rows, int n, int k) {
  (void)rows; (void)n; (void)k;
  return kStatusBytes;
}

size_t sv_prune_workspace_bytes(int B, int N, int k) {
  (void)B; (void)N; (void)k;
  return kStatusBytes;
}

size_t sv_retrieve_workspace_bytes(int B, int H, int n_kv_heads, int head_dim, int n_vis, int k) {
  (void)H; (void)head_dim; (void)k;
  if (B < 0 || n_kv_heads < 0 || n_vis < 0) return kStatusBytes;
  // status | per-row completion counters [B][Hkv] | scores [B][Hkv][n_vis]
  return kStatusBytes + round256((size_t)B * n_kv_heads * sizeof(int)) +
         round256((size_t)B * n_kv_heads * n_vis * sizeof(float));
}

size_t sv_attn_workspace_bytes(int B, int H, int n_kv_heads, int head_dim, int n_tokens) {
  if (B < 0 || H <= 0 || n_kv_heads <= 0 || head_dim <= 0 || n_tokens < 0 || H % n_kv_heads)
    return kStatusBytes;
  const int G = H / n_kv_heads;
  const sv::AttnPlan p = sv::attn_plan(B, n_kv_heads, G, n_tokens);
  const size_t parts = (size_t)B * n_kv_heads * p.nsplit_max * G;
  // status | per-(sequence, KV head) split counters | (m, l) partials | o partials
  return kStatusBytes + round256((size_t)B * n_kv_heads * sizeof(int)) + round256(parts * 2 * sizeof(float)) +
         round256(parts * head_dim * sizeof(float));
}

size_t sv_evict_workspace_bytes(void) { return kStatusBytes; }

int sv_retrieve_kernel_count(int batch, int n_kv_heads, int n_vis) {
  if (n_vis <= 0) return 0;
  return sv::retrieve_fuses_topk(batch * n_kv_heads, n_vis) ? 1 : 2;
}

int sv_attn_kernel_count(int B, int H, int n_kv_heads, int n_tokens) {
  if (B <= 0 || H <= 0 || n_kv_heads <= 0 || H % n_kv_heads || n_tokens <= 0) return 0;
  return sv::attn_kernel_count(B, n_kv_heads, H / n_kv_heads, n_tokens);
}

// ------------------------------------------------------------------ prefill

sv_status sv_salience_prefill(const void* q, const void* k, int B, int H, int N, int d, float scale,
                              float* salience, void* ws, size_t ws_bytes, void* stream) {
  if (!q || !k || !salience) return fail(SV_ERR_INVALID_ARG, "q, k and salience must be non-NULL");
  if (B < 0 || H <= 0 || N <= 0) return fail(SV_ERR_INVALID_ARG, "need B >= 0, H > 0, N > 0");
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(SV_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (!sv::salience_head_dim_supported(d))
    return fail(SV_ERR_UNSUPPORTED, "salience head_dim %d (64, 72, 80 or 128)", d);
  if (!aligned16(q) || !aligned16(k)) return fail(SV_ERR_INVALID_ARG, "q and k must be 16-byte aligned");
  if (N > (1 << 24)) return fail(SV_ERR_UNSUPPORTED, "N = %d > 2^24 tokens", N);
  if ((long long)B * H * ((N + 127) / 128) > 0x7fffffffLL) return fail(SV_ERR_INVALID_ARG, "B * H * N too large");
  sv_status s = check_ws(ws, ws_bytes, sv_salience_workspace_bytes(B, H, N, d));
  if (s != SV_OK) return s;
  if (B == 0) return SV_OK;
  cudaError_t e = sv::launch_salience(q, k, B, H, N, d, scale, salience, after_status(ws),
                                      status_word(ws), num_sms(), static_cast<cudaStream_t>(stream));
  if (e == cudaErrorInvalidValue)
    return fail(SV_ERR_CUDA, "tensor-map encoding or launch rejected the salience operands");
  return cuda_status(e, "sv_salience_prefill");
}

size_t sv_salience_summary_workspace_bytes(int B, int H, int N, int d, int R) {
  (void)d;
  (void)R;
  if (B < 0 || H < 0 || N < 0) return kStatusBytes;
  return kStatusBytes + round256((size_t)B * H * N * sizeof(float));
}

sv_status sv_salience_summary(const void* q, const void* k, int B, int H, int N, int d, int R, float scale,
                              float* salience, void* ws, size_t ws_bytes, void* stream) {
  if (!q || !k || !salience) return fail(SV_ERR_INVALID_ARG, "q, k and salience must be non-NULL");
  if (B < 0 || H <= 0 || N <= 0) return fail(SV_ERR_INVALID_ARG, "need B >= 0, H > 0, N > 0");
  if (R < 1 || R > 16 || R > N) return fail(SV_ERR_INVALID_ARG, "need 1 <= R <= min(16, N) (R = %d)", R);
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(SV_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (d < 8 || d > 256 || d % 8) return fail(SV_ERR_UNSUPPORTED, "summary salience head_dim %d (multiple of 8, <= 256)", d);
  if (!aligned16(q) || !aligned16(k)) return fail(SV_ERR_INVALID_ARG, "q and k must be 16-byte aligned");
  if (sv::summary_smem_bytes(N, d, R) > kMaxSmemPerBlock - 4096)
    return fail(SV_ERR_UNSUPPORTED, "R * N = %d logits do not fit in shared memory", R * N);
  if ((long long)B * H > 0x7fffffffLL) return fail(SV_ERR_INVALID_ARG, "B * H too large");
  sv_status s = check_ws(ws, ws_bytes, sv_salience_summary_workspace_bytes(B, H, N, d, R));
  if (s != SV_OK) return s;
  if (B == 0) return SV_OK;
  cudaError_t e = sv::launch_summary_salience(q, k, B, H, N, d, R, scale, salience,
                                              reinterpret_cast<float*>(after_status(ws)),
                                              static_cast<cudaStream_t>(stream));
  return cuda_status(e, "sv_salience_summary");
}

sv_status sv_topk_rows(const float* scores, int rows, int n, int k, int32_t* idx, void* ws,
                       size_t ws_bytes, void* stream) {
  if (!scores || !idx) return fail(SV_ERR_INVALID_ARG, "scores and idx must be non-NULL");
  if (rows < 0 || n <= 0 || n > (1 << 24)) return fail(SV_ERR_INVALID_ARG, "need rows >= 0, 0 < n <= 2^24");
  if (k < 1 || k > n) return fail(SV_ERR_INVALID_ARG, "need 1 <= k <= n (k = %d, n = %d)", k, n);
  sv_status s = check_ws(ws, ws_bytes, sv_topk_workspace_bytes(rows, n, k));
  if (s != SV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // long rows: a cluster of CTAs per row; otherwise one CTA per row
  const cudaError_t e = sv::topk_prefers_cluster(n)
                            ? sv::launch_topk_cluster(scores, rows, n, k, idx, st)
                            : sv::launch_topk_rows(scores, rows, n, k, idx, st);
  return cuda_status(e, "sv_topk_rows");
}

sv_status sv_prune_threshold(const float* salience, int B, int N, float threshold, const void* feat,
                             int64_t row_bytes, void* feat_out, int32_t* kept_idx, int32_t* kept_count,
                             void* ws, size_t ws_bytes, void* stream) {
  if (!salience || !kept_idx || !kept_count)
    return fail(SV_ERR_INVALID_ARG, "salience, kept_idx and kept_count must be non-NULL");
  if (B < 0 || N <= 0 || N > (1 << 24)) return fail(SV_ERR_INVALID_ARG, "need B >= 0, 0 < N <= 2^24");
  if (std::isnan(threshold)) return fail(SV_ERR_INVALID_ARG, "threshold is NaN");
  if (row_bytes < 0 || row_bytes % 16) return fail(SV_ERR_INVALID_ARG, "row_bytes must be a multiple of 16");
  if (row_bytes > 0 && (!feat || !feat_out)) return fail(SV_ERR_INVALID_ARG, "feat and feat_out must be non-NULL");
  if (row_bytes > 0 && (!aligned16(feat) || !aligned16(feat_out)))
    return fail(SV_ERR_INVALID_ARG, "feat and feat_out must be 16-byte aligned");
  sv_status s = check_ws(ws, ws_bytes, sv_prune_workspace_bytes(B, N, 1));
  if (s != SV_OK) return s;
  if (B == 0) return SV_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = sv::launch_threshold_select(salience, B, N, threshold, kept_idx, kept_count, st);
  if (e == cudaSuccess && row_bytes > 0)
    e = sv::launch_gather_rows(feat, B, N, N, row_bytes, kept_idx, feat_out, status_word(ws), st, kept_count);
  return cuda_status(e, "sv_prune_threshold");
}

sv_status sv_prune_compact(const float* salience, int B, int N, int k, const void* feat,
                           int64_t row_bytes, void* feat_out, int32_t* kept_idx, void* ws,
                           size_t ws_bytes, void* stream) {
  if (!salience || !kept_idx) return fail(SV_ERR_INVALID_ARG, "salience and kept_idx must be non-NULL");
  if (B < 0 || N <= 0 || N > (1 << 24)) return fail(SV_ERR_INVALID_ARG, "need B >= 0, 0 < N <= 2^24");
  if (k < 1 || k > N) return fail(SV_ERR_INVALID_ARG, "need 1 <= k <= N (k = %d, N = %d)", k, N);
  if (row_bytes < 0 || row_bytes % 16) return fail(SV_ERR_INVALID_ARG, "row_bytes must be a multiple of 16");
  if (row_bytes > 0 && (!feat || !feat_out)) return fail(SV_ERR_INVALID_ARG, "feat and feat_out must be non-NULL");
  if (row_bytes > 0 && (!aligned16(feat) || !aligned16(feat_out)))
    return fail(SV_ERR_INVALID_ARG, "feat and feat_out must be 16-byte aligned");
  sv_status s = check_ws(ws, ws_bytes, sv_prune_workspace_bytes(B, N, k));
  if (s != SV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = sv::launch_topk_rows(salience, B, N, k, kept_idx, st);
  if (e == cudaSuccess && row_bytes > 0)
    e = sv::launch_gather_rows(feat, B, N, k, row_bytes, kept_idx, feat_out, status_word(ws), st);
  return cuda_status(e, "sv_prune_compact");
}

// ------------------------------------------------------------------ decode

sv_status sv_retrieve_topk(const void* q, int R, int H, const sv_kv_layer* layer,
                           const sv_seq_batch* seqs, int k, int32_t* vis_idx, float* scores,
                           void* ws, size_t ws_bytes, void* stream) {
  sv_status s = sv::check_retrieve_args(q, R, H, layer, seqs, k, vis_idx);
  if (s != SV_OK) return s;
  const int Hkv = layer->n_kv_heads;
  s = check_ws(ws, ws_bytes, sv_retrieve_workspace_bytes(seqs->batch, H, Hkv, layer->head_dim, seqs->n_vis, k));
  if (s != SV_OK) return s;
  if (seqs->batch == 0) return SV_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t rows = (size_t)seqs->batch * Hkv;
  int* row_done = reinterpret_cast<int*>(after_status(ws));
  float* sc = scores ? scores : reinterpret_cast<float*>(after_status(ws) + round256(rows * sizeof(int)));
  cudaError_t e = sv::launch_retrieve(q, R, H, H / Hkv, layer->k_pool, layer->num_blocks, Hkv,
                                      layer->head_dim, seqs->block_table, seqs->max_blocks, seqs->n_vis,
                                      seqs->batch, sc, status_word(ws), num_sms(), row_done, k, vis_idx, st,
                                      lens_of(seqs), seqs->n_text);
  return cuda_status(e, "sv_retrieve_topk");
}

size_t sv_retrieve_softmax_workspace_bytes(int B, int R, int H, int n_kv_heads, int head_dim, int n_vis,
                                           int n_text) {
  if (B < 0 || R <= 0 || H <= 0 || n_kv_heads <= 0 || H % n_kv_heads || n_vis < 0 || n_text < 0) return kStatusBytes;
  return kStatusBytes + sv::retrieve_softmax_workspace_bytes(B, R, H, n_kv_heads, head_dim, n_vis, n_text);
}

sv_status sv_retrieve_topk_softmax(const void* q, int R, int H, float scale, const sv_kv_layer* layer,
                                   const sv_seq_batch* seqs, const float* lse, int k, int32_t* vis_idx,
                                   float* scores, void* ws, size_t ws_bytes, void* stream) {
  sv_status s = check_cache(layer, seqs, false);
  if (s != SV_OK) return s;
  s = reject_lens(seqs, "sv_retrieve_topk_softmax");
  if (s != SV_OK) return s;
  if (!q || !vis_idx) return fail(SV_ERR_INVALID_ARG, "q and vis_idx must be non-NULL");
  if (!aligned16(q)) return fail(SV_ERR_INVALID_ARG, "q must be 16-byte aligned");
  const int Hkv = layer->n_kv_heads;
  if (R <= 0 || H <= 0 || H % Hkv) return fail(SV_ERR_INVALID_ARG, "need R > 0 and H a multiple of n_kv_heads");
  if (R * (H / Hkv) > sv::retrieve_softmax_max_rows())
    return fail(SV_ERR_UNSUPPORTED, "R * (H / n_kv_heads) = %d > %d question rows per KV head", R * (H / Hkv),
                sv::retrieve_softmax_max_rows());
  if (!(scale > 0.f) || !std::isfinite(scale)) return fail(SV_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (seqs->n_vis <= 0) return fail(SV_ERR_INVALID_ARG, "no visual tokens to retrieve from");
  if (k < 1 || k > seqs->n_vis) return fail(SV_ERR_INVALID_ARG, "need 1 <= k <= n_vis (k = %d)", k);
  s = check_ws(ws, ws_bytes,
               sv_retrieve_softmax_workspace_bytes(seqs->batch, R, H, Hkv, layer->head_dim, seqs->n_vis, seqs->n_text));
  if (s != SV_OK) return s;
  if (seqs->batch == 0) return SV_OK;
  cudaError_t e = sv::launch_retrieve_softmax(q, R, H, scale, layer->k_pool, layer->num_blocks, Hkv, layer->head_dim,
                                              seqs->block_table, seqs->max_blocks, seqs->n_vis, seqs->n_text,
                                              seqs->batch, lse, k, vis_idx, scores, after_status(ws), status_word(ws),
                                              static_cast<cudaStream_t>(stream));
  return cuda_status(e, "sv_retrieve_topk_softmax");
}

}  // extern "C"

// sv_sparse_decode_attn, and with k_new / v_new the fused append of one token
// per sequence before it (sv_decode_append_attn)
static sv_status decode_attn(const char* name, const void* q, int H, float scale, const sv_kv_layer* layer,
                             const sv_seq_batch* seqs, const void* k_new, const void* v_new,
                             const int32_t* vis_idx, int k, void* out, float* lse, void* ws, size_t ws_bytes,
                             void* stream) {
  sv_status s = check_cache(layer, seqs, true);
  if (s != SV_OK) return s;
  if (!q || !out) return fail(SV_ERR_INVALID_ARG, "q and out must be non-NULL");
  if (!aligned16(q)) return fail(SV_ERR_INVALID_ARG, "q must be 16-byte aligned");
  const int Hkv = layer->n_kv_heads;
  if (H <= 0 || H % Hkv) return fail(SV_ERR_INVALID_ARG, "H must be a positive multiple of n_kv_heads");
  if (H / Hkv > 16) return fail(SV_ERR_UNSUPPORTED, "query heads per KV head %d > 16", H / Hkv);
  if (!std::isfinite(scale)) return fail(SV_ERR_INVALID_ARG, "scale must be finite");
  const bool append = k_new != nullptr || v_new != nullptr;
  if (append) {
    if (!k_new || !v_new) return fail(SV_ERR_INVALID_ARG, "k_new and v_new must be non-NULL");
    if (!aligned16(k_new) || !aligned16(v_new))
      return fail(SV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if ((long long)seqs->n_vis + seqs->n_text + 1 > (long long)seqs->max_blocks * SV_BLOCK_TOKENS)
      return fail(SV_ERR_INVALID_ARG, "appending a token overflows the block table");
  }
  const int k_vis = vis_idx ? k : seqs->n_vis;
  if (vis_idx && (k < 0 || k > seqs->n_vis)) return fail(SV_ERR_INVALID_ARG, "need 0 <= k <= n_vis");
  const int n_tok = k_vis + seqs->n_text + (append ? 1 : 0);
  if (n_tok <= 0) return fail(SV_ERR_INVALID_ARG, "the attended token set is empty");
  s = check_ws(ws, ws_bytes, sv_attn_workspace_bytes(seqs->batch, H, Hkv, layer->head_dim, n_tok));
  if (s != SV_OK) return s;
  if (seqs->batch == 0) return SV_OK;
  const sv::AttnPlan p = sv::attn_plan(seqs->batch, Hkv, H / Hkv, n_tok);
  const size_t parts = (size_t)seqs->batch * Hkv * p.nsplit * (H / Hkv);
  sv::AttnArgs a;
  a.q = q; a.H = H; a.scale = scale;
  a.k_pool = layer->k_pool; a.v_pool = layer->v_pool;
  a.num_blocks = layer->num_blocks; a.Hkv = Hkv; a.D = layer->head_dim;
  a.block_table = seqs->block_table; a.max_blocks = seqs->max_blocks;
  a.vis_idx = vis_idx; a.k_vis = k_vis; a.n_vis = seqs->n_vis; a.n_text = seqs->n_text;
  a.batch = seqs->batch; a.out = out; a.lse = lse;
  a.lens = lens_of(seqs);
  a.k_new = k_new; a.v_new = v_new;
  // the counters' offset depends only on the batch shape, so a workspace
  // reused with other token counts finds them where the last call zeroed them
  const size_t cnt_bytes = round256((size_t)seqs->batch * Hkv * sizeof(int));
  a.split_done = reinterpret_cast<int*>(after_status(ws));
  a.part_ml = reinterpret_cast<float*>(after_status(ws) + cnt_bytes);
  a.part_o = reinterpret_cast<float*>(after_status(ws) + cnt_bytes + round256(parts * 2 * sizeof(float)));
  a.status = status_word(ws);
  return cuda_status(sv::launch_sparse_attn(a, static_cast<cudaStream_t>(stream)), name);
}

extern "C" {

sv_status sv_sparse_decode_attn(const void* q, int H, float scale, const sv_kv_layer* layer,
                                const sv_seq_batch* seqs, const int32_t* vis_idx, int k, void* out,
                                float* lse, void* ws, size_t ws_bytes, void* stream) {
  return decode_attn("sv_sparse_decode_attn", q, H, scale, layer, seqs, nullptr, nullptr, vis_idx, k, out, lse, ws,
                     ws_bytes, stream);
}

sv_status sv_decode_append_attn(const void* q, int H, float scale, const sv_kv_layer* layer,
                                const sv_seq_batch* seqs, const void* k_new, const void* v_new,
                                const int32_t* vis_idx, int k, void* out, float* lse, void* ws, size_t ws_bytes,
                                void* stream) {
  if (!k_new || !v_new) return fail(SV_ERR_INVALID_ARG, "k_new and v_new must be non-NULL");
  return decode_attn("sv_decode_append_attn", q, H, scale, layer, seqs, k_new, v_new, vis_idx, k, out, lse, ws,
                     ws_bytes, stream);
}

// ------------------------------------------------------------------ rounds

sv_status sv_pack_kv(const sv_kv_layer* src, const sv_seq_batch* seqs, const int32_t* vis_idx, int k,
                     const sv_kv_layer* dst, const sv_seq_batch* dst_seqs, void* ws, size_t ws_bytes,
                     void* stream) {
  sv_status s = check_cache(src, seqs, true);
  if (s != SV_OK) return s;
  s = check_cache(dst, dst_seqs, true);
  if (s != SV_OK) return s;
  s = reject_lens(seqs, "sv_pack_kv");
  if (s == SV_OK) s = reject_lens(dst_seqs, "sv_pack_kv");
  if (s != SV_OK) return s;
  if (dst->n_kv_heads != src->n_kv_heads || dst->head_dim != src->head_dim)
    return fail(SV_ERR_INVALID_ARG, "source and packed layers differ in n_kv_heads or head_dim");
  if (dst->k_pool == src->k_pool || dst->v_pool == src->v_pool)
    return fail(SV_ERR_INVALID_ARG, "the packed layer must not share pools with the source");
  const int k_vis = vis_idx ? k : seqs->n_vis;
  if (vis_idx && (k < 0 || k > seqs->n_vis)) return fail(SV_ERR_INVALID_ARG, "need 0 <= k <= n_vis");
  if (dst_seqs->batch != seqs->batch || dst_seqs->n_vis != k_vis || dst_seqs->n_text != seqs->n_text)
    return fail(SV_ERR_INVALID_ARG,
                "packed batch must have the source's batch, n_vis = k (%d) and n_text = %d", k_vis, seqs->n_text);
  s = check_ws(ws, ws_bytes, sv_evict_workspace_bytes());
  if (s != SV_OK) return s;
  cudaError_t e = sv::launch_pack_kv(src->k_pool, src->v_pool, src->num_blocks, seqs->block_table,
                                     seqs->max_blocks, seqs->n_vis, vis_idx, k_vis, seqs->n_text, dst->k_pool,
                                     dst->v_pool, dst->num_blocks, dst_seqs->block_table, dst_seqs->max_blocks,
                                     seqs->batch, src->n_kv_heads, src->head_dim, status_word(ws),
                                     static_cast<cudaStream_t>(stream));
  return cuda_status(e, "sv_pack_kv");
}

sv_status sv_evict_qa_tokens(const sv_kv_layer* layers, int n_layers, sv_seq_batch* seqs,
                             int32_t text_begin, int32_t text_end, int32_t* n_blocks_in_use,
                             void* ws, size_t ws_bytes, void* stream) {
  if (!layers || !seqs || n_layers < 0) return fail(SV_ERR_INVALID_ARG, "layers and seqs must be non-NULL");
  if (reject_lens(seqs, "sv_evict_qa_tokens") != SV_OK) return SV_ERR_UNSUPPORTED;
  if (text_begin < 0 || text_begin > text_end || text_end > seqs->n_text)
    return fail(SV_ERR_INVALID_ARG, "need 0 <= text_begin <= text_end <= n_text (%d, %d, %d)",
                text_begin, text_end, seqs->n_text);
  for (int l = 0; l < n_layers; ++l) {
    sv_status s = check_cache(&layers[l], seqs, true);
    if (s != SV_OK) return s;
  }
  sv_status s = check_ws(ws, ws_bytes, sv_evict_workspace_bytes());
  if (s != SV_OK) return s;
  const int count = seqs->n_text - text_end;   // later text tokens to move down
  if (text_end > text_begin && count > 0) {
    for (int l = 0; l < n_layers; ++l) {
      cudaError_t e = sv::launch_kv_move_down(
          layers[l].k_pool, layers[l].v_pool, layers[l].num_blocks, layers[l].n_kv_heads,
          layers[l].head_dim, seqs->block_table, seqs->max_blocks, seqs->batch,
          seqs->n_vis + text_begin, seqs->n_vis + text_end, count, status_word(ws),
          static_cast<cudaStream_t>(stream));
      if (e != cudaSuccess) return cuda_status(e, "sv_evict_qa_tokens");
    }
  }
  seqs->n_text -= text_end - text_begin;
  if (n_blocks_in_use) {
    const int need = (seqs->n_vis + seqs->n_text + SV_BLOCK_TOKENS - 1) / SV_BLOCK_TOKENS;
    for (int b = 0; b < seqs->batch; ++b) n_blocks_in_use[b] = need;
  }
  return SV_OK;
}

sv_status sv_kv_append(const sv_kv_layer* layer, const sv_seq_batch* seqs, const void* k_new,
                       const void* v_new, int T, void* ws, size_t ws_bytes, void* stream) {
  sv_status s = check_cache(layer, seqs, true);
  if (s != SV_OK) return s;
  if (T < 0) return fail(SV_ERR_INVALID_ARG, "T must be >= 0");
  if (T > 0 && (!k_new || !v_new)) return fail(SV_ERR_INVALID_ARG, "k_new and v_new must be non-NULL");
  if (T > 0 && (!aligned16(k_new) || !aligned16(v_new)))
    return fail(SV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
  if ((long long)seqs->n_vis + seqs->n_text + T > (long long)seqs->max_blocks * SV_BLOCK_TOKENS)
    return fail(SV_ERR_INVALID_ARG, "appending %d tokens overflows the block table", T);
  s = check_ws(ws, ws_bytes, sv_evict_workspace_bytes());
  if (s != SV_OK) return s;
  return cuda_status(sv::launch_kv_append(layer->k_pool, layer->v_pool, layer->num_blocks,
                                          layer->n_kv_heads, layer->head_dim, seqs->block_table,
                                          seqs->max_blocks, seqs->batch, seqs->n_vis + seqs->n_text,
                                          k_new, v_new, T, status_word(ws),
                                          static_cast<cudaStream_t>(stream), lens_of(seqs), seqs->n_vis,
                                          seqs->n_text),
                     "sv_kv_append");
}

sv_status sv_read_device_status(void* ws, int clear, int32_t* status_out, void* stream) {
  if (!ws || !status_out) return fail(SV_ERR_INVALID_ARG, "ws and status_out must be non-NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(ws, 0, sizeof(int32_t), st);
  if (e != cudaSuccess) return cuda_status(e, "sv_read_device_status");
  *status_out = v;
  return SV_OK;
}

}  // extern "C"
