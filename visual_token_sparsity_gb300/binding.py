"""ctypes binding of libsv (include/sv.h): argument marshalling only.

Every function here has the name of the C entry point it calls, checks that
tensors have the dtype / layout the C ABI documents, passes raw device
pointers and raises :class:`SvError` on a non-OK status.  All arithmetic runs
in the library's CUDA kernels; there is no other implementation behind these
calls, and loading fails loudly when the library is missing.
"""

import ctypes
import os

import torch

from . import build as _build

_lib = None

SV_OK = 0
SV_DEV_BAD_BLOCK = 0x1
SV_DEV_BAD_INDEX = 0x2
SV_DEV_BAD_LENGTH = 0x4
BLOCK_TOKENS = 16


class SvError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"sv status {status}: {msg}")
        self.status = status


class sv_kv_layer(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32)]


class sv_seq_batch(ctypes.Structure):
    _fields_ = [("block_table", ctypes.c_void_p), ("batch", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("n_vis", ctypes.c_int32),
                ("n_text", ctypes.c_int32), ("n_vis_seq", ctypes.c_void_p),
                ("n_text_seq", ctypes.c_void_p), ("k_seq", ctypes.c_void_p)]


_VP, _SZ, _I, _F, _I64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_float, ctypes.c_int64
_SIGS = {
    "sv_status_string": (ctypes.c_char_p, [_I]),
    "sv_last_error": (ctypes.c_char_p, []),
    "sv_version": (ctypes.c_char_p, []),
    "sv_salience_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "sv_retrieve_kernel_count": (_I, [_I, _I, _I]),
    "sv_salience_kernel_count": (_I, [_I, _I]),
    "sv_attn_kernel_count": (_I, [_I, _I, _I, _I]),
    "sv_topk_workspace_bytes": (_SZ, [_I, _I, _I]),
    "sv_prune_workspace_bytes": (_SZ, [_I, _I, _I]),
    "sv_retrieve_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "sv_attn_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "sv_evict_workspace_bytes": (_SZ, []),
    "sv_salience_prefill": (_I, [_VP, _VP, _I, _I, _I, _I, _F, _VP, _VP, _SZ, _VP]),
    "sv_topk_rows": (_I, [_VP, _I, _I, _I, _VP, _VP, _SZ, _VP]),
    "sv_prune_compact": (_I, [_VP, _I, _I, _I, _VP, _I64, _VP, _VP, _VP, _SZ, _VP]),
    "sv_retrieve_topk": (_I, [_VP, _I, _I, ctypes.POINTER(sv_kv_layer),
                              ctypes.POINTER(sv_seq_batch), _I, _VP, _VP, _VP, _SZ, _VP]),
    "sv_retrieve_topk_noalloc": (_I, [_VP, _I, _I, ctypes.POINTER(sv_kv_layer),
                                      ctypes.POINTER(sv_seq_batch), _I, _VP, _VP, _VP]),
    "sv_sparse_decode_attn": (_I, [_VP, _I, _F, ctypes.POINTER(sv_kv_layer),
                                   ctypes.POINTER(sv_seq_batch), _VP, _I, _VP, _VP, _VP, _SZ, _VP]),
    "sv_decode_append_attn": (_I, [_VP, _I, _F, ctypes.POINTER(sv_kv_layer), ctypes.POINTER(sv_seq_batch),
                                   _VP, _VP, _VP, _I, _VP, _VP, _VP, _SZ, _VP]),
    "sv_evict_qa_tokens": (_I, [ctypes.POINTER(sv_kv_layer), _I, ctypes.POINTER(sv_seq_batch),
                                ctypes.c_int32, ctypes.c_int32, _VP, _VP, _SZ, _VP]),
    "sv_kv_append": (_I, [ctypes.POINTER(sv_kv_layer), ctypes.POINTER(sv_seq_batch), _VP, _VP, _I,
                          _VP, _SZ, _VP]),
    "sv_pack_kv": (_I, [ctypes.POINTER(sv_kv_layer), ctypes.POINTER(sv_seq_batch), _VP, _I,
                        ctypes.POINTER(sv_kv_layer), ctypes.POINTER(sv_seq_batch), _VP, _SZ, _VP]),
    "sv_salience_summary_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "sv_salience_summary": (_I, [_VP, _VP, _I, _I, _I, _I, _I, ctypes.c_float, _VP, _VP, _SZ, _VP]),
    "sv_prune_threshold": (_I, [_VP, _I, _I, ctypes.c_float, _VP, ctypes.c_int64, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "sv_retrieve_softmax_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "sv_retrieve_topk_softmax": (_I, [_VP, _I, _I, ctypes.c_float, ctypes.POINTER(sv_kv_layer),
                                      ctypes.POINTER(sv_seq_batch), _VP, _I, _VP, _VP, _VP, _SZ, _VP]),
    "sv_read_device_status": (_I, [_VP, _I, ctypes.POINTER(ctypes.c_int32), _VP]),
}
EXPORTED = tuple(_SIGS)


def library_path():
    return _build.LIB


def load(path=None):
    """Load libsv.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libsv.so is not built ({path}); run visual_token_sparsity_gb300.build")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(status):
    if status != SV_OK:
        raise SvError(status, _lib.sv_last_error().decode())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _ws(ws):
    return _ptr(ws, torch.uint8, "ws"), ctypes.c_size_t(ws.numel())


def workspace(nbytes, device="cuda"):
    """Zero-filled device workspace of ``nbytes`` bytes (status word cleared)."""
    return torch.zeros(int(nbytes), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ descriptors

class KvLayer:
    """One layer's paged cache: bf16 pools [num_blocks][Hkv][16][d]."""

    def __init__(self, k_pool, v_pool):
        assert k_pool.shape == v_pool.shape and k_pool.shape[2] == BLOCK_TOKENS
        self.k_pool, self.v_pool = k_pool, v_pool
        self.c = sv_kv_layer(_ptr(k_pool, torch.bfloat16, "k_pool"), _ptr(v_pool, torch.bfloat16, "v_pool"),
                             k_pool.shape[0], k_pool.shape[1], k_pool.shape[3])


class SeqBatch:
    """Block table (int32 [batch][max_blocks]) plus lengths: uniform n_vis /
    n_text, or -- with the optional int32 [batch] device tensors n_vis_seq,
    n_text_seq, k_seq -- per-sequence counts, n_vis / n_text then being the
    capacities."""

    def __init__(self, block_table, n_vis, n_text, n_vis_seq=None, n_text_seq=None, k_seq=None):
        self.block_table = block_table
        self.n_vis_seq, self.n_text_seq, self.k_seq = n_vis_seq, n_text_seq, k_seq
        B = block_table.shape[0]

        def opt(t, name):
            if t is None:
                return None
            if t.shape != (B,):
                raise ValueError(f"{name} must have shape ({B},), got {tuple(t.shape)}")
            return _ptr(t, torch.int32, name)
        self.c = sv_seq_batch(_ptr(block_table, torch.int32, "block_table"), B,
                              block_table.shape[1], int(n_vis), int(n_text), opt(n_vis_seq, "n_vis_seq"),
                              opt(n_text_seq, "n_text_seq"), opt(k_seq, "k_seq"))

    @property
    def n_vis(self):
        return self.c.n_vis

    @property
    def n_text(self):
        return self.c.n_text

    @n_text.setter
    def n_text(self, v):
        self.c.n_text = int(v)


# ------------------------------------------------------------------ sizes

def sv_salience_workspace_bytes(B, H, N, d):
    return load().sv_salience_workspace_bytes(B, H, N, d)


def sv_topk_workspace_bytes(rows, n, k):
    return load().sv_topk_workspace_bytes(rows, n, k)


def sv_prune_workspace_bytes(B, N, k):
    return load().sv_prune_workspace_bytes(B, N, k)


def sv_retrieve_workspace_bytes(B, H, n_kv_heads, head_dim, n_vis, k):
    return load().sv_retrieve_workspace_bytes(B, H, n_kv_heads, head_dim, n_vis, k)


def sv_attn_workspace_bytes(B, H, n_kv_heads, head_dim, n_tokens):
    return load().sv_attn_workspace_bytes(B, H, n_kv_heads, head_dim, n_tokens)


def sv_evict_workspace_bytes():
    return load().sv_evict_workspace_bytes()


def sv_salience_kernel_count(N, d):
    """Kernels one sv_salience_prefill call launches (3, or 4 for long sequences)."""
    return load().sv_salience_kernel_count(int(N), int(d))


def sv_retrieve_kernel_count(batch, n_kv_heads, n_vis):
    """Kernels one sv_retrieve_topk call launches (1: fused top-k, 2: separate top-k)."""
    return load().sv_retrieve_kernel_count(int(batch), int(n_kv_heads), int(n_vis))


def sv_attn_kernel_count(B, H, n_kv_heads, n_tokens):
    """Kernels one sv_sparse_decode_attn call launches (1: fused split merge, 2: merge kernel)."""
    return load().sv_attn_kernel_count(int(B), int(H), int(n_kv_heads), int(n_tokens))


# ------------------------------------------------------------------ calls

def sv_salience_prefill(q, k, scale, salience, ws, stream=None):
    """q, k: bf16 [B][H][N][d]; salience: fp32 [B][N] (written)."""
    lib = load()
    B, H, N, d = q.shape
    assert k.shape == q.shape and salience.shape == (B, N)
    _check(lib.sv_salience_prefill(_ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), B, H, N, d,
                                   float(scale), _ptr(salience, torch.float32, "salience"), *_ws(ws),
                                   _stream(stream)))


def sv_salience_summary_workspace_bytes(B, H, N, d, R):
    return load().sv_salience_summary_workspace_bytes(B, H, N, d, R)


def sv_salience_summary(q, k, R, scale, salience, ws, stream=None):
    """q, k: bf16 [B][H][N][d] (summary tokens first); salience: fp32 [B][N] (written)."""
    lib = load()
    B, H, N, d = q.shape
    assert k.shape == q.shape and salience.shape == (B, N)
    _check(lib.sv_salience_summary(_ptr(q, torch.bfloat16, "q"), _ptr(k, torch.bfloat16, "k"), B, H, N, d, int(R),
                                   float(scale), _ptr(salience, torch.float32, "salience"), *_ws(ws),
                                   _stream(stream)))


def sv_prune_threshold(salience, threshold, feat, feat_out, kept_idx, kept_count, ws, stream=None):
    """salience fp32 [B][N]; feat / feat_out [B][N][...] rows (or None); kept_idx int32 [B][N];
    kept_count int32 [B] (device)."""
    lib = load()
    B, N = salience.shape
    row_bytes = 0 if feat is None else feat.shape[2] * feat.element_size()
    _check(lib.sv_prune_threshold(_ptr(salience, torch.float32, "salience"), B, N, float(threshold),
                                  _ptr(feat, None, "feat"), row_bytes, _ptr(feat_out, None, "feat_out"),
                                  _ptr(kept_idx, torch.int32, "kept_idx"), _ptr(kept_count, torch.int32, "kept_count"),
                                  *_ws(ws), _stream(stream)))


def sv_topk_rows(scores, k, idx, ws, stream=None):
    """scores: fp32 [rows][n]; idx: int32 [rows][k] (written, ascending)."""
    lib = load()
    rows, n = scores.shape
    assert idx.shape == (rows, k)
    _check(lib.sv_topk_rows(_ptr(scores, torch.float32, "scores"), rows, n, k,
                            _ptr(idx, torch.int32, "idx"), *_ws(ws), _stream(stream)))


def sv_prune_compact(salience, k, feat, feat_out, kept_idx, ws, stream=None):
    """salience fp32 [B][N]; feat [B][N][C] (any dtype); feat_out [B][k][C]; kept_idx int32 [B][k]."""
    lib = load()
    B, N = salience.shape
    row_bytes = 0 if feat is None else feat.shape[2] * feat.element_size()
    _check(lib.sv_prune_compact(_ptr(salience, torch.float32, "salience"), B, N, k,
                                _ptr(feat, None, "feat"), row_bytes, _ptr(feat_out, None, "feat_out"),
                                _ptr(kept_idx, torch.int32, "kept_idx"), *_ws(ws), _stream(stream)))


def sv_retrieve_topk(q, layer, seqs, k, vis_idx, scores, ws, stream=None):
    """q bf16 [B][R][H][d]; vis_idx int32 [B][Hkv][k]; scores fp32 [B][Hkv][n_vis] or None."""
    lib = load()
    B, R, H, d = q.shape
    _check(lib.sv_retrieve_topk(_ptr(q, torch.bfloat16, "q"), R, H, ctypes.byref(layer.c),
                                ctypes.byref(seqs.c), k, _ptr(vis_idx, torch.int32, "vis_idx"),
                                _ptr(scores, torch.float32, "scores"), *_ws(ws), _stream(stream)))


def sv_retrieve_softmax_workspace_bytes(B, R, H, n_kv_heads, head_dim, n_vis, n_text):
    return load().sv_retrieve_softmax_workspace_bytes(B, R, H, n_kv_heads, head_dim, n_vis, n_text)


def sv_retrieve_topk_softmax(q, scale, layer, seqs, k, vis_idx, scores, ws, lse=None, stream=None):
    """q bf16 [B][R][H][d]; lse fp32 [B][R][H] (natural log) or None; vis_idx int32 [B][Hkv][k]."""
    lib = load()
    B, R, H, d = q.shape
    _check(lib.sv_retrieve_topk_softmax(_ptr(q, torch.bfloat16, "q"), R, H, float(scale), ctypes.byref(layer.c),
                                        ctypes.byref(seqs.c), _ptr(lse, torch.float32, "lse"), int(k),
                                        _ptr(vis_idx, torch.int32, "vis_idx"), _ptr(scores, torch.float32, "scores"),
                                        *_ws(ws), _stream(stream)))


def sv_retrieve_topk_noalloc(q, layer, seqs, k, vis_idx, scores=None, stream=None):
    """As sv_retrieve_topk, for callers that cannot allocate: no workspace; the
    library's fixed device scratch holds the scores (limit B * Hkv * n_vis <= 2^21)."""
    lib = load()
    B, R, H, d = q.shape
    _check(lib.sv_retrieve_topk_noalloc(_ptr(q, torch.bfloat16, "q"), R, H, ctypes.byref(layer.c),
                                        ctypes.byref(seqs.c), k, _ptr(vis_idx, torch.int32, "vis_idx"),
                                        _ptr(scores, torch.float32, "scores"), _stream(stream)))


def sv_sparse_decode_attn(q, scale, layer, seqs, vis_idx, k, out, lse, ws, stream=None):
    """q bf16 [B][H][d]; vis_idx int32 [B][Hkv][k] or None; out bf16 [B][H][d]; lse fp32 [B][H] or None."""
    lib = load()
    B, H, d = q.shape
    _check(lib.sv_sparse_decode_attn(_ptr(q, torch.bfloat16, "q"), H, float(scale), ctypes.byref(layer.c),
                                     ctypes.byref(seqs.c), _ptr(vis_idx, torch.int32, "vis_idx"), k,
                                     _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
                                     *_ws(ws), _stream(stream)))


def sv_decode_append_attn(q, scale, layer, seqs, k_new, v_new, vis_idx, k, out, lse, ws, stream=None):
    """sv_kv_append of one token (k_new, v_new bf16 [B][Hkv][d]) then sparse attention over it and the
    cache, in one launch; n_text unchanged (the caller adds 1)."""
    lib = load()
    B, H, d = q.shape
    _check(lib.sv_decode_append_attn(_ptr(q, torch.bfloat16, "q"), H, float(scale), ctypes.byref(layer.c),
                                     ctypes.byref(seqs.c), _ptr(k_new, torch.bfloat16, "k_new"),
                                     _ptr(v_new, torch.bfloat16, "v_new"), _ptr(vis_idx, torch.int32, "vis_idx"),
                                     k, _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
                                     *_ws(ws), _stream(stream)))


def sv_evict_qa_tokens(layers, seqs, text_begin, text_end, ws, stream=None):
    """Evicts text span [text_begin, text_end) in every layer; returns pages in use per sequence."""
    lib = load()
    arr = (sv_kv_layer * len(layers))(*[l.c for l in layers])
    used = (ctypes.c_int32 * max(1, seqs.c.batch))()
    _check(lib.sv_evict_qa_tokens(arr, len(layers), ctypes.byref(seqs.c), int(text_begin), int(text_end),
                                  ctypes.cast(used, ctypes.c_void_p), *_ws(ws), _stream(stream)))
    return list(used)[: seqs.c.batch]


def sv_kv_append(layer, seqs, k_new, v_new, ws, stream=None):
    """k_new, v_new bf16 [B][T][Hkv][d] written at positions n_vis + n_text ...; n_text unchanged."""
    lib = load()
    T = k_new.shape[1]
    _check(lib.sv_kv_append(ctypes.byref(layer.c), ctypes.byref(seqs.c), _ptr(k_new, torch.bfloat16, "k_new"),
                            _ptr(v_new, torch.bfloat16, "v_new"), T, *_ws(ws), _stream(stream)))


def sv_pack_kv(src, seqs, vis_idx, k, dst, dst_seqs, ws, stream=None):
    """Copy the selected visual (vis_idx int32 [B][Hkv][k], or None = all) and all
    text K/V rows of src to positions [0, k + n_text) of dst (see include/sv.h)."""
    lib = load()
    _check(lib.sv_pack_kv(ctypes.byref(src.c), ctypes.byref(seqs.c), _ptr(vis_idx, torch.int32, "vis_idx"), int(k),
                          ctypes.byref(dst.c), ctypes.byref(dst_seqs.c), *_ws(ws), _stream(stream)))


def sv_read_device_status(ws, clear=False, stream=None):
    lib = load()
    out = ctypes.c_int32(0)
    _check(lib.sv_read_device_status(_ptr(ws, torch.uint8, "ws"), 1 if clear else 0, ctypes.byref(out),
                                     _stream(stream)))
    return out.value
