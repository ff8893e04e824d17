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
// host-side shadow, not device memory); every call looks up the device
// address with cudaGetSymbolAddress on the current device.  The lookup is
// cheap once the module is loaded, and it stays right if the context is
// destroyed and recreated (the array may then sit at another address).  With
// lazy module loading the first lookup on a device loads this module and
// maps the array, which can fail when device memory is exhausted.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>

#include "../../include/sv.h"
#include "api_checks.h"
#include "kernels.h"

namespace {

constexpr size_t kStatusBytes = 256;
constexpr size_t kMaxScores = size_t(1) << 21;                  // fp32 scores: 8 MiB
constexpr size_t kNoAllocScratchBytes = kStatusBytes + kMaxScores * sizeof(float);

// [0, 256): device status word; [256, ...): scores [B][Hkv][n_vis].
static __device__ __align__(256) unsigned char g_scratch[kNoAllocScratchBytes];

sv_status noalloc_fail(sv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  sv::set_error_message(buf);
  return s;
}

// Device address of g_scratch in the current device's context.
sv_status scratch_on_current_device(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
  if (e != cudaSuccess || !p)
    return noalloc_fail(SV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
  *out = p;
  return SV_OK;
}

}  // namespace

extern "C" sv_status sv_retrieve_topk_noalloc(const void* q, int R, int H, const sv_kv_layer* layer,
                                              const sv_seq_batch* seqs, int k, int32_t* vis_idx,
                                              float* scores, void* stream) {
  // the checks of sv_retrieve_topk, so both entry points accept the same calls
  sv_status s = sv::check_retrieve_args(q, R, H, layer, seqs, k, vis_idx);
  if (s != SV_OK) return s;
  const int Hkv = layer->n_kv_heads;
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
  s = scratch_on_current_device(&base);
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
