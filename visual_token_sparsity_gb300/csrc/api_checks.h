// Host-side argument checks shared by the C-ABI entry points of libsv that
// live in different translation units (api.cu, noalloc.cu), so that calls
// documented to compute the same thing accept and reject the same inputs.
#pragma once

#include "../../include/sv.h"

namespace sv {

// Records `msg` as this thread's sv_last_error() text.
void set_error_message(const char* msg);

// The layer / batch descriptors of a paged cache: non-NULL, 16-byte aligned
// pools, supported head_dim, 32-bit row ids, lengths within the block table.
sv_status check_cache(const sv_kv_layer* layer, const sv_seq_batch* seqs, bool need_v);

// Everything sv_retrieve_topk checks except its workspace.
sv_status check_retrieve_args(const void* q, int R, int H, const sv_kv_layer* layer, const sv_seq_batch* seqs,
                              int k, const int32_t* vis_idx);

}  // namespace sv
