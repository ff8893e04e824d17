// sv_retrieve_topk_noalloc: query-aware retrieval without a caller workspace.
//
// Some callers cannot allocate device memory at all: a plugin that runs
// inside a host framework which owns every byte of device memory through its
// own pool, or a latency-critical loop in which cudaMalloc (which may
// synchronise the device and take driver locks) is not allowed.  They cannot
// provide the scores workspace that sv_retrieve_topk needs.  This variant runs
// the same scoring kernel and top-k routine (here as two kernels: paged
// scoring GEMV, then row top-k) with the scores kept in a fixed scratch array
// that lives in this library's device image.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds its kNoAllocScratchBytes until the process exits.  Host code
// must not pass the variable's name to a kernel (on the host it names a
// host-side shadow, not device memory); the device address is looked up once
// per device with cudaGetSymbolAddress, with that device current, on the first
// call made on it.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>

#include "../../include/sv.h"
#include "kernels.h"

namespace sv {
void set_error_message(const char* msg);
}  // namespace sv

namespace {

constexpr size_t kStatusBytes = 256;
constexpr size_t kMaxScores = size_t(1) << 21;                  // fp32 scores: 8 MiB
constexpr size_t kNoAllocScratchBytes = kStatusBytes + kMaxScores * sizeof(float);
constexpr int kMaxDevices = 64;

// [0, 256): device status word; [256, ...): scores [B][Hkv][n_vis].
static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

void* g_scratch_addr[kMaxDevices] = {};

sv_status noalloc_fail(sv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  sv::set_error_message(buf);
  return s;
}

// Device address of g_scratch on the current device (set up on first use).
sv_status scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return noalloc_fail(SV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return noalloc_fail(SV_ERR_UNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess || !p)
      return noalloc_fail(SV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SV_OK;
}

}  // namespace

extern "C" sv_status sv_retrieve_topk_noalloc(const void* q, int R, int H, const sv_kv_layer* layer,
                                              const sv_seq_batch* seqs, int k, int32_t* vis_idx,
                                              float* scores, void* stream) {
  if (!layer || !seqs) return noalloc_fail(SV_ERR_INVALID_ARG, "layer or batch descriptor is NULL");
  if (!q || !vis_idx || !layer->k_pool || !seqs->block_table)
    return noalloc_fail(SV_ERR_INVALID_ARG, "q, vis_idx, k_pool and block_table must be non-NULL");
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(layer->k_pool)) & 15u)
    return noalloc_fail(SV_ERR_INVALID_ARG, "q and k_pool must be 16-byte aligned");
  if (layer->head_dim != 64 && layer->head_dim != 128)
    return noalloc_fail(SV_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", layer->head_dim);
  const int Hkv = layer->n_kv_heads;
  if (layer->num_blocks <= 0 || Hkv <= 0) return noalloc_fail(SV_ERR_INVALID_ARG, "num_blocks and n_kv_heads must be positive");
  if (R <= 0 || H <= 0 || H % Hkv) return noalloc_fail(SV_ERR_INVALID_ARG, "need R > 0 and H a multiple of n_kv_heads");
  if (seqs->batch < 0 || seqs->max_blocks <= 0 || seqs->n_vis <= 0 || seqs->n_text < 0)
    return noalloc_fail(SV_ERR_INVALID_ARG, "need batch >= 0, max_blocks > 0, n_vis > 0, n_text >= 0");
  if ((long long)seqs->n_vis + seqs->n_text > (long long)seqs->max_blocks * SV_BLOCK_TOKENS)
    return noalloc_fail(SV_ERR_INVALID_ARG, "n_vis + n_text exceeds max_blocks * 16");
  if (k < 1 || k > seqs->n_vis) return noalloc_fail(SV_ERR_INVALID_ARG, "need 1 <= k <= n_vis (k = %d)", k);
  const size_t n_scores = (size_t)seqs->batch * Hkv * seqs->n_vis;
  if (n_scores > kMaxScores)
    return noalloc_fail(SV_ERR_WORKSPACE,
                        "batch * n_kv_heads * n_vis = %zu exceeds the fixed scratch of %zu scores "
                        "(use sv_retrieve_topk with a workspace)", n_scores, kMaxScores);
  if (seqs->batch == 0) return SV_OK;

  sv::SeqLens lens;
  lens.n_vis = seqs->n_vis_seq;
  lens.n_text = seqs->n_text_seq;
  lens.k = seqs->k_seq;
  void* base = nullptr;
  sv_status s = scratch_on_current_device(&base);
  if (s != SV_OK) return s;
  int* status = static_cast<int*>(base);
  float* sc = scores ? scores : reinterpret_cast<float*>(static_cast<char*>(base) + kStatusBytes);
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), st);   // the status word starts at zero
  if (e == cudaSuccess) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    e = sv::launch_retrieve(q, R, H, H / Hkv, layer->k_pool, layer->num_blocks, Hkv, layer->head_dim,
                            seqs->block_table, seqs->max_blocks, seqs->n_vis, seqs->batch, sc, status, sms,
                            nullptr, k, vis_idx, st, lens, seqs->n_text);
  }
  if (e != cudaSuccess) return noalloc_fail(SV_ERR_CUDA, "sv_retrieve_topk_noalloc: %s", cudaGetErrorString(e));
  return SV_OK;
}
