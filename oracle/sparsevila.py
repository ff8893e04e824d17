"""fp64 restatement of what the SparseVILA hot path computes.

TEST INFRASTRUCTURE ONLY (see the package docstring): the product path never
imports this module.

Conventions shared with the library (all of them layout, not arithmetic):

* Query head ``h`` reads KV head ``h // G`` with ``G = H // Hkv`` (grouped-query
  attention: consecutive query heads share one KV head).
* A sequence's cache holds its visual tokens at logical positions
  ``[0, n_vis)`` and its text tokens after them.
* The paged cache stores token ``t`` of sequence ``b`` in block
  ``block_table[b, t // 16]`` at row ``t % 16``; a pool is laid out
  ``[num_blocks][Hkv][16][d]``.
* Top-k keeps the k largest scores; equal scores are broken towards the lower
  index; the kept indices are returned in ascending order.

Inputs are float64 arrays holding the exact values of the bf16 tensors the GPU
reads (bf16 -> fp64 is exact).
"""

import math

import numpy as np

BLOCK_TOKENS = 16


def _as_f64(x):
    return np.asarray(x, dtype=np.float64)


def salience(q, k, scale=None):
    """Query-agnostic salience of every encoder token.

    velog.io summary §3.1 (encoder-type table, "no summary token" row for
    SigLIP / QwenVL): a token's importance is the intra-visual attention it
    receives, averaged over all tokens.  xllm-io review §三 gives it as
    Salience(t) = (1/N) * sum over the other tokens of their attention to t.
    The reading taken: per head, row-softmax the scaled logits
    Z = scale * Q K^T (row i = the attending token), take the mean of column j
    over the N rows, then average over the H heads.

    q, k: [B][H][N][d].  Returns s: [B][N] with s[b].sum() == 1.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    s = np.zeros((B, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            z = scale * (q[b, h] @ k[b, h].T)             # [N query][N key]
            z = z - z.max(axis=1, keepdims=True)
            p = np.exp(z)
            p = p / p.sum(axis=1, keepdims=True)           # row-stochastic
            s[b] += p.sum(axis=0)                          # attention received
    return s / (H * N)


def summary_salience(q, k, R, scale=None):
    """Query-agnostic salience for encoders with summary tokens.

    velog.io summary §3.1 (encoder-type table): with a single summary token
    (CLIP) a token's importance is the attention it contributes to the global
    embedding, i.e. the summary token's attention to it; with several
    summary tokens (RADIO) it is the mean attention toward them.  Reading
    taken: the R summary tokens are the first R tokens of the sequence; per
    head, the summary rows of the row-softmax of Z = scale * Q K^T (softmax
    over all N tokens) are averaged over the R rows and the H heads.

    q, k: [B][H][N][d].  Returns s: [B][N] with s[b].sum() == 1.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    s = np.zeros((B, N), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            z = scale * (q[b, h, :R] @ k[b, h].T)         # [R summary rows][N keys]
            z = z - z.max(axis=1, keepdims=True)
            p = np.exp(z)
            p = p / p.sum(axis=1, keepdims=True)
            s[b] += p.sum(axis=0)
    return s / (H * R)


def topk_ascending(scores, k):
    """Indices of the k largest entries of every row, in ascending order.

    velog.io summary §3.1 (drop the tokens of lowest aggregate salience) and
    §3.2 (activate the highest-scoring tokens); xllm-io review §五
    (``torch.topk(scores, top_k)``).  Ties go to the lower index.

    scores: [..., n].  Returns int64 [..., k].
    """
    scores = _as_f64(scores)
    lead = scores.shape[:-1]
    n = scores.shape[-1]
    if not 0 <= k <= n:
        raise ValueError("k out of range")
    flat = scores.reshape(-1, n)
    out = np.empty((flat.shape[0], k), dtype=np.int64)
    pos = np.arange(n)
    for r in range(flat.shape[0]):
        order = np.lexsort((pos, -flat[r]))   # score descending, index ascending
        out[r] = np.sort(order[:k])
    return out.reshape(lead + (k,))


def prune_compact(sal, feat, k):
    """Prefill prune: keep the k most salient tokens and gather their rows.

    velog.io summary §2 table ("prefill: query-agnostic pruning ... actually
    deleted") and §3.1; xllm-io review §五 ``query_agnostic_pruning`` (keeps the
    tokens that pass the salience cut).  Kept rows stay in token order.

    sal: [B][N]; feat: [B][N][...] of any dtype.  Returns (idx [B][k],
    feat_out [B][k][...]).
    """
    idx = topk_ascending(sal, k)
    feat = np.asarray(feat)
    out = np.stack([feat[b, idx[b]] for b in range(feat.shape[0])])
    return idx, out


def prune_threshold(sal, feat, threshold):
    """Prefill prune by a salience threshold (a variable count per frame).

    xllm-io review §五 query_agnostic_pruning: tokens whose salience exceeds
    the threshold are kept (strictly greater), in their original order, and
    their rows are gathered.

    sal: [B][N]; feat: [B][N][C].  Returns a list over frames of
    (kept indices ascending, kept rows [count][C]).
    """
    sal = np.asarray(sal)
    feat = np.asarray(feat)
    out = []
    for b in range(sal.shape[0]):
        idx = np.array([j for j in range(sal.shape[1]) if sal[b, j] > threshold], dtype=np.int64)
        out.append((idx, feat[b, idx]))
    return out


def paged_view(pool, block_table, n_tokens):
    """Logical [B][Hkv][n_tokens][d] view of one layer's paged pool.

    Layout only (the pages fix no cache layout): token t of sequence b is row
    t % 16 of block block_table[b, t // 16].
    """
    pool = np.asarray(pool)
    bt = np.asarray(block_table)
    B = bt.shape[0]
    _, Hkv, bs, d = pool.shape
    assert bs == BLOCK_TOKENS
    out = np.empty((B, Hkv, n_tokens, d), dtype=pool.dtype)
    for b in range(B):
        for t in range(n_tokens):
            out[b, :, t, :] = pool[bt[b, t // BLOCK_TOKENS], :, t % BLOCK_TOKENS, :]
    return out


def retrieval_scores(q, k_vis):
    """Query-aware relevance of every cached visual key.

    velog.io summary §3.2 "Query-Aware Token Selection": the current turn's text
    query is the Query, the cached vision tokens are the Keys, and the
    aggregate attention strength between them ranks the tokens.  xllm-io review
    §三 Selected = TopK(Query . KV_Cache, k) and §五
    ``matmul(query, keys.T)``.  Reading taken: the raw dot product, summed over
    the query rows and over the query heads that share the KV head.

    q: [B][R][H][d]; k_vis: [B][Hkv][Nv][d].  Returns [B][Hkv][Nv].
    """
    q = _as_f64(q)
    k_vis = _as_f64(k_vis)
    B, R, H, d = q.shape
    Hkv = k_vis.shape[1]
    G = H // Hkv
    out = np.zeros(k_vis.shape[:3], dtype=np.float64)
    for b in range(B):
        for g in range(Hkv):
            for r in range(R):
                for h in range(g * G, (g + 1) * G):
                    out[b, g] += k_vis[b, g] @ q[b, r, h]
    return out


def retrieve_topk(q, k_vis, k):
    """Retrieval scores followed by the per-KV-head top-k (see above).

    velog.io summary §3.2: high-scoring tokens stay active for decoding; the
    others remain cached but inactive.  Returns (idx [B][Hkv][k], scores).
    """
    sc = retrieval_scores(q, k_vis)
    return topk_ascending(sc, k), sc


def retrieval_scores_softmax(q, K, n_vis, n_text, scale=None, lse=None):
    """Softmax-normalised query-aware relevance of every cached visual token.

    velog.io summary §3.2 "Query-Aware Token Selection": the aggregated
    attention strength between the question's rows (Query) and the cached
    vision tokens (Key); the retrieval kernel there runs alongside the
    question's FlashAttention-2 prefill.  Reading taken for this variant:
    the attention probability of each question row and query head to visual
    token j, normalised over every cached token (visual and text, no causal
    mask), summed over the rows and the heads that share the KV head.  When
    ``lse`` is given (a caller's own prefill attention statistics, natural
    log, [B][R][H]) it is used as each row's normaliser instead.

    q: [B][R][H][d]; K: logical [B][Hkv][>= n_vis + n_text][d].
    Returns [B][Hkv][n_vis].
    """
    q = _as_f64(q)
    K = _as_f64(K)
    B, R, H, d = q.shape
    Hkv = K.shape[1]
    G = H // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, Hkv, n_vis), dtype=np.float64)
    for b in range(B):
        for g in range(Hkv):
            for r in range(R):
                for h in range(g * G, (g + 1) * G):
                    z = scale * (K[b, g, :n_vis + n_text] @ q[b, r, h])
                    if lse is None:
                        m = z.max()
                        norm = m + math.log(np.exp(z - m).sum())
                    else:
                        norm = float(lse[b, r, h])
                    out[b, g] += np.exp(z[:n_vis] - norm)
    return out


def sparse_decode_attention(q, K, V, vis_idx, n_vis, n_text, scale=None):
    """Decode attention over the retrieved visual tokens plus all text tokens.

    velog.io summary §3.2 (only the query-relevant subset of the preserved
    visual cache is read) and §4.5 kernel table ("decoding attention" over the
    reduced KV).  Softmax attention is written out directly over the token set
    T = vis_idx[b, g] U [n_vis, n_vis + n_text).

    q: [B][H][d]; K, V: logical [B][Hkv][>= n_vis + n_text][d];
    vis_idx: [B][Hkv][k] or None (= every visual token).
    Returns (out [B][H][d], lse [B][H]) with lse = log sum_t exp(scale q.k_t).
    """
    q = _as_f64(q)
    K = _as_f64(K)
    V = _as_f64(V)
    B, H, d = q.shape
    Hkv = K.shape[1]
    G = H // Hkv
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((B, H, d), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    text = np.arange(n_vis, n_vis + n_text, dtype=np.int64)
    for b in range(B):
        for h in range(H):
            g = h // G
            vis = np.arange(n_vis) if vis_idx is None else np.asarray(vis_idx[b, g], dtype=np.int64)
            tokens = np.concatenate([vis, text])
            z = scale * (K[b, g, tokens] @ q[b, h])
            m = z.max()
            w = np.exp(z - m)
            out[b, h] = (w / w.sum()) @ V[b, g, tokens]
            lse[b, h] = m + math.log(w.sum())
    return out, lse


def pack_selected_kv(K, V, vis_idx, n_vis, n_text):
    """Pack-once KV: the retrieved visual tokens and the text, contiguous.

    velog.io summary §3.2 (why decode-time selection is efficient): the
    selected KV entries are gathered into contiguous memory so the attention
    reads them with regular, coalesced accesses.  Per (sequence b, KV head g)
    the packed cache holds the selected visual tokens in vis_idx[b, g] order,
    then the n_text text tokens in their order.

    K, V: logical [B][Hkv][>= n_vis + n_text][d]; vis_idx: [B][Hkv][k] or None
    (= every visual token).  Returns logical K', V' [B][Hkv][k + n_text][d].
    """
    K = np.asarray(K)
    V = np.asarray(V)
    B, Hkv = K.shape[0], K.shape[1]
    k = n_vis if vis_idx is None else np.asarray(vis_idx).shape[2]
    Kp = np.empty((B, Hkv, k + n_text, K.shape[3]), dtype=K.dtype)
    Vp = np.empty_like(Kp)
    for b in range(B):
        for g in range(Hkv):
            vis = np.arange(n_vis) if vis_idx is None else np.asarray(vis_idx[b, g], dtype=np.int64)
            tokens = np.concatenate([vis, np.arange(n_vis, n_vis + n_text, dtype=np.int64)])
            Kp[b, g] = K[b, g, tokens]
            Vp[b, g] = V[b, g, tokens]
    return Kp, Vp


def evict_qa_tokens(K, V, n_vis, n_text, text_begin, text_end):
    """Partial KV-cache eviction between conversation rounds.

    velog.io summary §4.1 Setup (information leakage): after each round only
    the previous question/answer KV entries are removed and the visual cache is
    kept.  xllm-io review §五 ``partial_kv_cache_eviction`` keeps every visual
    entry and every entry outside the evicted Q&A.  Here the Q&A is the
    text-relative span [text_begin, text_end).

    K, V: logical [B][Hkv][>= n_vis + n_text][d].  Returns (K', V', n_text').
    """
    K = np.asarray(K)
    V = np.asarray(V)
    keep = []
    for p in range(n_vis + n_text):
        is_visual = p < n_vis
        in_qa = (not is_visual) and text_begin <= p - n_vis < text_end
        if is_visual or not in_qa:
            keep.append(p)
    keep = np.asarray(keep, dtype=np.int64)
    return K[:, :, keep], V[:, :, keep], len(keep) - n_vis


def append_tokens(K, V, n_used, k_new, v_new):
    """Append new tokens' K/V after the first n_used logical positions.

    k_new, v_new: [B][T][Hkv][d] (token-major, as a projection writes them).
    Returns logical K', V' of length n_used + T.
    """
    K = np.asarray(K)[:, :, :n_used]
    V = np.asarray(V)[:, :, :n_used]
    kn = np.transpose(np.asarray(k_new), (0, 2, 1, 3))
    vn = np.transpose(np.asarray(v_new), (0, 2, 1, 3))
    return np.concatenate([K, kn], axis=2), np.concatenate([V, vn], axis=2)
