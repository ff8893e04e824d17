"""Pins of the fp64 oracle against closed forms, invariants, brute force and
library routines.  CPU only.

Each test is chosen so that a plausible slip in the oracle (row mean instead of
column mean, a sum instead of a mean over heads, a wrong GQA head->group map, a
dropped query row, an off-by-one in the evicted span, a wrong tie-break) fails.
"""

import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from visual_token_sparsity_gb300 import synth

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- salience

def test_salience_rows_stochastic_sum_to_one():
    q = RNG.standard_normal((2, 3, 17, 8))
    k = RNG.standard_normal((2, 3, 17, 8))
    s = oracle.salience(q, k)
    np.testing.assert_allclose(s.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert (s > 0).all()


def test_summary_salience_single_row_is_torch_softmax_row():
    q = RNG.standard_normal((2, 3, 9, 4))
    k = RNG.standard_normal((2, 3, 9, 4))
    s = oracle.summary_salience(q, k, 1)
    zt = torch.einsum("bhd,bhnd->bhn", torch.from_numpy(q[:, :, 0]), torch.from_numpy(k)) / 2.0
    ref = torch.softmax(zt, dim=-1).mean(dim=1).numpy()          # head mean of the CLS row
    np.testing.assert_allclose(s, ref, rtol=0, atol=1e-14)


def test_summary_salience_all_rows_is_full_salience_and_rows_sum_to_one():
    q = RNG.standard_normal((1, 2, 7, 3))
    k = RNG.standard_normal((1, 2, 7, 3))
    np.testing.assert_allclose(oracle.summary_salience(q, k, 7), oracle.salience(q, k), rtol=0, atol=1e-14)
    s = oracle.summary_salience(q, k, 3)
    np.testing.assert_allclose(s.sum(-1), 1.0, rtol=0, atol=1e-13)


def test_summary_salience_uses_only_leading_rows_and_zero_query_is_uniform():
    q = RNG.standard_normal((1, 2, 6, 4))
    k = RNG.standard_normal((1, 2, 6, 4))
    q2 = q.copy()
    q2[:, :, 2:] = RNG.standard_normal((1, 2, 4, 4))                # non-summary rows do not matter
    np.testing.assert_array_equal(oracle.summary_salience(q, k, 2), oracle.summary_salience(q2, k, 2))
    q3 = q.copy()
    q3[:, :, :2] = 0.0
    np.testing.assert_allclose(oracle.summary_salience(q3, k, 2), 1.0 / 6, rtol=0, atol=1e-15)


def test_salience_zero_query_is_uniform():
    k = RNG.standard_normal((1, 2, 11, 4))
    s = oracle.salience(np.zeros_like(k), k)
    np.testing.assert_allclose(s, 1.0 / 11, rtol=0, atol=1e-15)


def test_salience_equal_keys_is_uniform():
    q = RNG.standard_normal((1, 2, 9, 4))
    k = np.broadcast_to(RNG.standard_normal(4), (1, 2, 9, 4)).copy()
    np.testing.assert_allclose(oracle.salience(q, k), 1.0 / 9, rtol=0, atol=1e-15)


def _magnet_head(N, d, j, c, u):
    """All queries equal u; key j equals c*u; other keys zero."""
    q = np.tile(u, (N, 1))
    k = np.zeros((N, d))
    k[j] = c * u
    return q, k


def test_salience_magnet_closed_form_column_not_row():
    # Every query puts weight e^a / (e^a + N - 1) on key j and 1/(e^a+N-1) on
    # the others, so the attention *received* by j is that weight; a row mean
    # would give 1/N everywhere.
    N, d = 7, 4
    u = np.array([1.0, -0.5, 0.25, 2.0])
    qa, ka = _magnet_head(N, d, j=2, c=0.75, u=u)
    qb, kb = _magnet_head(N, d, j=5, c=-1.5, u=u)
    q = np.stack([qa, qb])[None]
    k = np.stack([ka, kb])[None]
    scale = 0.3
    s = oracle.salience(q, k, scale=scale)
    uu = float(u @ u)
    expect = np.zeros(N)
    for j, c in ((2, 0.75), (5, -1.5)):
        a = scale * c * uu
        z = math.exp(a) + N - 1
        head = np.full(N, 1.0 / z)
        head[j] = math.exp(a) / z
        expect += head / 2.0          # mean over the 2 heads
    np.testing.assert_allclose(s[0], expect, rtol=1e-13, atol=0)


def test_salience_default_scale_is_inverse_sqrt_d():
    q = RNG.standard_normal((1, 1, 6, 9))
    k = RNG.standard_normal((1, 1, 6, 9))
    np.testing.assert_allclose(oracle.salience(q, k), oracle.salience(q, k, scale=1 / 3.0),
                               rtol=1e-14)


def test_salience_token_permutation_equivariant():
    q = RNG.standard_normal((1, 2, 10, 5))
    k = RNG.standard_normal((1, 2, 10, 5))
    perm = RNG.permutation(10)
    s = oracle.salience(q, k)
    sp = oracle.salience(q[:, :, perm], k[:, :, perm])
    np.testing.assert_allclose(sp[0], s[0, perm], rtol=1e-13)
    # permuting only the attending (query) tokens changes nothing
    np.testing.assert_allclose(oracle.salience(q[:, :, perm], k), s, rtol=1e-13)


def test_salience_brute_force_tiny():
    # Scalar loops over (h, i, j), independent of the matrix code path.
    H, N, d = 2, 5, 3
    q = RNG.standard_normal((1, H, N, d))
    k = RNG.standard_normal((1, H, N, d))
    sc = 0.7
    s = [0.0] * N
    for h in range(H):
        for i in range(N):
            logits = [sc * sum(q[0, h, i, e] * k[0, h, j, e] for e in range(d)) for j in range(N)]
            den = sum(math.exp(x) for x in logits)
            for j in range(N):
                s[j] += math.exp(logits[j]) / den / (H * N)
    np.testing.assert_allclose(oracle.salience(q, k, scale=sc)[0], s, rtol=1e-12)


# ---------------------------------------------------------------- top-k

def _brute_topk(row, k):
    """The unique k-subset whose members all beat all non-members under
    (score descending, index ascending)."""
    n = len(row)
    found = []
    for sub in itertools.combinations(range(n), k):
        chosen = set(sub)
        ok = all((row[a] > row[b]) or (row[a] == row[b] and a < b)
                 for a in chosen for b in range(n) if b not in chosen)
        if ok:
            found.append(list(sub))
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("n", [1, 4, 7])
def test_topk_brute_force_with_ties(n):
    for trial in range(20):
        row = RNG.integers(-2, 3, size=n).astype(np.float64)   # many ties
        for k in range(n + 1):
            got = oracle.topk_ascending(row[None], k)[0].tolist()
            assert got == _brute_topk(row, k)


def test_topk_matches_torch_topk_on_distinct_values():
    x = RNG.standard_normal((5, 300))
    for k in (1, 37, 150, 300):
        got = oracle.topk_ascending(x, k)
        ref = torch.topk(torch.from_numpy(x), k, dim=-1).indices.sort(-1).values.numpy()
        np.testing.assert_array_equal(got, ref)


def test_topk_signed_zero_ties_to_lower_index():
    row = np.array([-0.0, 0.0, -1.0, 0.0])
    assert oracle.topk_ascending(row[None], 1)[0].tolist() == [0]
    assert oracle.topk_ascending(row[None], 2)[0].tolist() == [0, 1]


def test_topk_permutation_equivariant():
    x = RNG.standard_normal(50)
    perm = RNG.permutation(50)
    a = set(oracle.topk_ascending(x[None], 12)[0].tolist())
    b = set(perm[oracle.topk_ascending(x[perm][None], 12)[0]].tolist())
    assert a == b


def test_prune_compact_gathers_kept_rows():
    sal = np.array([[0.1, 0.5, 0.2, 0.5, 0.05]])
    feat = np.arange(5 * 3).reshape(1, 5, 3).astype(np.uint16)
    idx, out = oracle.prune_compact(sal, feat, 3)
    assert idx[0].tolist() == [1, 2, 3]
    np.testing.assert_array_equal(out[0], feat[0, [1, 2, 3]])


# ---------------------------------------------------------------- retrieval

def test_retrieval_identity_keys_give_summed_query():
    B, R, H, Hkv, d = 1, 3, 4, 2, 6
    q = RNG.standard_normal((B, R, H, d))
    k = np.broadcast_to(np.eye(d), (B, Hkv, d, d)).copy()     # key j = e_j
    sc = oracle.retrieval_scores(q, k)
    for g in range(Hkv):
        expect = q[0, :, 2 * g:2 * g + 2].sum(axis=(0, 1))
        np.testing.assert_allclose(sc[0, g], expect, rtol=1e-14)


def test_retrieval_head_to_group_is_floor_division():
    q = np.zeros((1, 1, 4, 3))
    q[0, 0, 1] = 1.0                                          # head 1 -> group 0
    k = RNG.standard_normal((1, 2, 5, 3))
    sc = oracle.retrieval_scores(q, k)
    np.testing.assert_allclose(sc[0, 0], k[0, 0].sum(-1), rtol=1e-14)
    np.testing.assert_array_equal(sc[0, 1], 0.0)


def test_retrieval_rows_are_linear_and_scale_free():
    q = RNG.standard_normal((2, 5, 6, 8))
    k = RNG.standard_normal((2, 3, 40, 8))
    one = q.sum(axis=1, keepdims=True)
    np.testing.assert_allclose(oracle.retrieval_scores(q, k), oracle.retrieval_scores(one, k),
                               rtol=1e-12, atol=1e-12)
    i1, _ = oracle.retrieve_topk(q, k, 10)
    i2, _ = oracle.retrieve_topk(2.5 * q, k, 10)
    np.testing.assert_array_equal(i1, i2)


def test_retrieval_ranking_equals_softmax_ranking_for_one_row_one_head():
    q = RNG.standard_normal((1, 1, 1, 16))
    k = RNG.standard_normal((1, 1, 64, 16))
    idx, sc = oracle.retrieve_topk(q, k, 16)
    p = torch.softmax(torch.from_numpy(sc[0, 0] / 4.0), dim=0).numpy()
    np.testing.assert_array_equal(idx[0, 0], np.sort(np.argsort(-p, kind="stable")[:16]))


# ---------------------------------------------------------------- attention

def _sdpa(q, K, V, scale):
    """torch scaled_dot_product_attention in fp64 with GQA head expansion."""
    B, H, d = q.shape
    G = H // K.shape[1]
    Kx = torch.from_numpy(K).repeat_interleave(G, dim=1)
    Vx = torch.from_numpy(V).repeat_interleave(G, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[:, :, None, :], Kx, Vx, scale=scale)
    return out[:, :, 0, :].numpy()


def test_softmax_retrieval_is_torch_softmax_mass_summed_over_rows_and_heads():
    B, R, H, Hkv, nv, nt, d = 2, 3, 4, 2, 11, 5, 8
    q = RNG.standard_normal((B, R, H, d))
    K = RNG.standard_normal((B, Hkv, nv + nt, d))
    got = oracle.retrieval_scores_softmax(q, K, nv, nt)
    Kt = torch.from_numpy(K).repeat_interleave(H // Hkv, dim=1)       # [B][H][n][d]
    p = torch.softmax(torch.einsum("brhd,bhnd->brhn", torch.from_numpy(q), Kt) / math.sqrt(d), dim=-1)
    ref = p[..., :nv].sum(dim=1).view(B, Hkv, H // Hkv, nv).sum(dim=2).numpy()
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def test_softmax_retrieval_mass_bounds_and_given_lse():
    B, R, H, Hkv, nv, nt, d = 1, 2, 6, 3, 9, 4, 4
    q = RNG.standard_normal((B, R, H, d))
    K = RNG.standard_normal((B, Hkv, nv + nt, d))
    sc = oracle.retrieval_scores_softmax(q, K, nv, nt)
    sc0 = oracle.retrieval_scores_softmax(q, K[:, :, :nv], nv, 0)       # no text: all mass is visual
    np.testing.assert_allclose(sc0.sum(-1), R * (H // Hkv), rtol=0, atol=1e-12)
    assert (sc.sum(-1) < sc0.sum(-1)).all()
    Kt = torch.from_numpy(K).repeat_interleave(H // Hkv, dim=1)
    lse = torch.logsumexp(torch.einsum("brhd,bhnd->brhn", torch.from_numpy(q), Kt) / math.sqrt(d), dim=-1).numpy()
    np.testing.assert_allclose(oracle.retrieval_scores_softmax(q, K, nv, nt, lse=lse), sc, rtol=1e-12, atol=0)
    np.testing.assert_allclose(oracle.retrieval_scores_softmax(q, K, nv, nt, lse=lse + 1.0), sc * math.exp(-1.0),
                               rtol=1e-12, atol=0)


def test_softmax_retrieval_one_row_one_head_ranks_like_dot_product():
    q = RNG.standard_normal((1, 1, 2, 6))
    K = RNG.standard_normal((1, 2, 30, 6))
    sm = oracle.retrieval_scores_softmax(q, K, 25, 5)
    raw = oracle.retrieval_scores(q, K[:, :, :25])
    for k in (1, 5, 24):
        np.testing.assert_array_equal(oracle.topk_ascending(sm.reshape(2, 25), k),
                                      oracle.topk_ascending(raw.reshape(2, 25), k))


def test_attention_all_tokens_equals_sdpa():
    B, H, Hkv, d, nv, nt = 2, 6, 2, 16, 30, 7
    q = RNG.standard_normal((B, H, d))
    K = RNG.standard_normal((B, Hkv, nv + nt, d))
    V = RNG.standard_normal((B, Hkv, nv + nt, d))
    out, lse = oracle.sparse_decode_attention(q, K, V, None, nv, nt, scale=0.25)
    np.testing.assert_allclose(out, _sdpa(q, K, V, 0.25), rtol=1e-12, atol=1e-12)
    # lse closed form via logsumexp
    Kx = np.repeat(K, 3, axis=1)
    z = 0.25 * np.einsum("bhd,bhtd->bht", q, Kx)
    np.testing.assert_allclose(lse, np.log(np.exp(z).sum(-1)), rtol=1e-12)


def test_attention_subset_equals_sdpa_on_gathered_tokens():
    B, H, Hkv, d, nv, nt = 1, 4, 2, 8, 20, 5
    q = RNG.standard_normal((B, H, d))
    K = RNG.standard_normal((B, Hkv, nv + nt, d))
    V = RNG.standard_normal((B, Hkv, nv + nt, d))
    idx = np.stack([np.sort(RNG.choice(nv, 6, replace=False)) for _ in range(Hkv)])[None]
    out, _ = oracle.sparse_decode_attention(q, K, V, idx, nv, nt, scale=0.5)
    for g in range(Hkv):
        tok = np.concatenate([idx[0, g], np.arange(nv, nv + nt)])
        ref = _sdpa(q[:, 2 * g:2 * g + 2], K[:, g:g + 1, tok], V[:, g:g + 1, tok], 0.5)
        np.testing.assert_allclose(out[:, 2 * g:2 * g + 2], ref, rtol=1e-12, atol=1e-12)
    # the order in which the visual indices are listed does not matter
    out2, _ = oracle.sparse_decode_attention(q, K, V, idx[:, :, ::-1], nv, nt, scale=0.5)
    np.testing.assert_allclose(out2, out, rtol=1e-13, atol=1e-13)


def test_attention_single_token_returns_its_value():
    q = RNG.standard_normal((1, 2, 4))
    K = RNG.standard_normal((1, 1, 1, 4))
    V = RNG.standard_normal((1, 1, 1, 4))
    out, lse = oracle.sparse_decode_attention(q, K, V, np.zeros((1, 1, 1), np.int64), 1, 0)
    np.testing.assert_allclose(out[0], np.repeat(V[0, 0], 2, axis=0), rtol=1e-15)
    np.testing.assert_allclose(lse[0], 0.5 * (q[0] @ K[0, 0, 0]), rtol=1e-13)


def test_attention_equal_keys_average_values_and_group_map():
    B, H, Hkv, d, nv, nt = 1, 4, 2, 3, 9, 3
    q = RNG.standard_normal((B, H, d))
    K = np.broadcast_to(RNG.standard_normal(d), (B, Hkv, nv + nt, d)).copy()
    V = RNG.standard_normal((B, Hkv, nv + nt, d))
    V[0, 1] += 100.0                                           # group 1 marked
    out, lse = oracle.sparse_decode_attention(q, K, V, None, nv, nt)
    for h in range(H):
        g = h // 2
        np.testing.assert_allclose(out[0, h], V[0, g].mean(0), rtol=1e-13)
    z = (q[0] @ K[0, 0, 0]) / math.sqrt(d)
    np.testing.assert_allclose(lse[0], z + math.log(nv + nt), rtol=1e-13)


# ---------------------------------------------------------------- eviction

def _logical(B=1, Hkv=2, n=12, d=2):
    # token position p holds value p in every entry: eviction results are
    # readable by eye
    x = np.broadcast_to(np.arange(n, dtype=np.float64)[None, None, :, None], (B, Hkv, n, d))
    return x.copy(), -x.copy()


def test_pack_all_visual_is_the_prefix_of_the_cache():
    K = RNG.standard_normal((2, 3, 13, 4))
    V = RNG.standard_normal((2, 3, 13, 4))
    Kp, Vp = oracle.pack_selected_kv(K, V, None, n_vis=9, n_text=3)
    np.testing.assert_array_equal(Kp, K[:, :, :12])
    np.testing.assert_array_equal(Vp, V[:, :, :12])


def test_pack_order_and_head_map_by_token_id_encoding():
    # every row encodes (sequence, head, token, tensor) so the packed rows can
    # be decoded back to where they came from
    B, Hkv, n_vis, n_text, d = 2, 3, 10, 4, 3
    K = np.zeros((B, Hkv, n_vis + n_text + 2, d))
    for b, g, t in itertools.product(range(B), range(Hkv), range(K.shape[2])):
        K[b, g, t] = (b, g, t)
    V = -K
    vis = np.stack([np.stack([np.sort(RNG.choice(n_vis, 4, replace=False)) for _ in range(Hkv)])
                    for _ in range(B)])
    Kp, Vp = oracle.pack_selected_kv(K, V, vis, n_vis, n_text)
    assert Kp.shape == (B, Hkv, 4 + n_text, d)
    for b, g in itertools.product(range(B), range(Hkv)):
        assert (Kp[b, g, :, 0] == b).all() and (Kp[b, g, :, 1] == g).all()
        assert list(Kp[b, g, :, 2]) == list(vis[b, g]) + list(range(n_vis, n_vis + n_text))
    np.testing.assert_array_equal(Vp, -Kp)


def test_threshold_prune_extremes_and_strictness():
    sal = np.array([[0.1, 0.3, 0.3, 0.05, 0.25]])
    feat = np.arange(5 * 2, dtype=np.float64).reshape(1, 5, 2)
    (idx, rows), = oracle.prune_threshold(sal, feat, -np.inf)
    assert list(idx) == [0, 1, 2, 3, 4] and (rows == feat[0]).all()
    (idx, rows), = oracle.prune_threshold(sal, feat, 0.3)            # equal to the threshold: dropped
    assert len(idx) == 0 and rows.shape == (0, 2)
    (idx, rows), = oracle.prune_threshold(sal, feat, 0.25)
    assert list(idx) == [1, 2] and (rows == feat[0, [1, 2]]).all()


@pytest.mark.parametrize("seed", range(5))
def test_threshold_prune_between_ranks_equals_topk(seed):
    rng = np.random.default_rng(seed)
    sal = rng.standard_normal((3, 40))
    feat = rng.standard_normal((3, 40, 4))
    for k in (1, 7, 39):
        srt = np.sort(sal, axis=1)[:, ::-1]
        for b in range(3):
            thr = 0.5 * (srt[b, k - 1] + srt[b, k])                  # between the k-th and (k+1)-th
            (idx, rows), = oracle.prune_threshold(sal[b:b + 1], feat[b:b + 1], thr)
            np.testing.assert_array_equal(idx, oracle.topk_ascending(sal[b:b + 1], k)[0])
            np.testing.assert_array_equal(rows, feat[b, idx])


def test_dense_attention_over_packed_equals_sparse_attention():
    B, H, Hkv, n_vis, n_text, d = 2, 6, 2, 20, 5, 8
    K = RNG.standard_normal((B, Hkv, n_vis + n_text, d))
    V = RNG.standard_normal((B, Hkv, n_vis + n_text, d))
    q = RNG.standard_normal((B, H, d))
    vis = np.stack([np.stack([np.sort(RNG.choice(n_vis, 7, replace=False)) for _ in range(Hkv)])
                    for _ in range(B)])
    ref, ref_lse = oracle.sparse_decode_attention(q, K, V, vis, n_vis, n_text)
    Kp, Vp = oracle.pack_selected_kv(K, V, vis, n_vis, n_text)
    got, got_lse = oracle.sparse_decode_attention(q, Kp, Vp, None, 7, n_text)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got_lse, ref_lse, rtol=0, atol=1e-12)


def test_evict_tail_span_truncates():
    K, V = _logical(n=12)
    K2, V2, nt = oracle.evict_qa_tokens(K, V, n_vis=5, n_text=7, text_begin=3, text_end=7)
    assert nt == 3
    assert K2[0, 0, :, 0].tolist() == [0, 1, 2, 3, 4, 5, 6, 7]
    np.testing.assert_array_equal(V2, -K2)


def test_evict_middle_span_moves_later_text_down():
    K, V = _logical(n=12)
    K2, _, nt = oracle.evict_qa_tokens(K, V, n_vis=5, n_text=7, text_begin=1, text_end=3)
    assert nt == 5
    assert K2[0, 1, :, 0].tolist() == [0, 1, 2, 3, 4, 5, 8, 9, 10, 11]


def test_evict_empty_span_and_full_text():
    K, V = _logical(n=12)
    K2, _, nt = oracle.evict_qa_tokens(K, V, 5, 7, 4, 4)
    assert nt == 7 and K2[0, 0, :, 0].tolist() == list(range(12))
    K3, _, nt3 = oracle.evict_qa_tokens(K, V, 5, 7, 0, 7)
    assert nt3 == 0 and K3[0, 0, :, 0].tolist() == list(range(5))


def test_append_then_evict_restores_cache():
    K, V = _logical(n=8)
    kn = RNG.standard_normal((1, 3, 2, 2))
    K2, V2 = oracle.append_tokens(K, V, 8, kn, -kn)
    assert K2.shape[2] == 11
    np.testing.assert_array_equal(K2[0, :, 8:], np.transpose(kn[0], (1, 0, 2)))
    K3, V3, nt = oracle.evict_qa_tokens(K2, V2, n_vis=5, n_text=6, text_begin=3, text_end=6)
    np.testing.assert_array_equal(K3, K)
    assert nt == 3


# ---------------------------------------------------------------- paging + recipe

def test_paged_view_inverts_pool_layout_for_any_table():
    B, Hkv, n, d = 2, 3, 37, 4
    x = torch.randn(B, Hkv, n, d, dtype=torch.float64)
    nb = synth.blocks_for(n)
    for identity in (True, False):
        bt = synth.random_block_table(B, nb + 1, 2 * (nb + 1) + 3, seed=7, identity=identity)
        pool = synth.scatter_to_pool(x, bt, 2 * (nb + 1) + 3)
        np.testing.assert_array_equal(oracle.paged_view(pool.numpy(), bt.numpy(), n), x.numpy())


def test_outlier_counts_follow_round_half_up():
    assert [synth.n_outliers(n) for n in (576, 729, 2880, 50176)] == [12, 15, 58, 1004]


def test_k_rounding_is_floor():
    assert synth.siglip_salience(keep=0.25).k == 182
    assert synth.siglip_salience(keep=0.5).k == 364
    assert synth.longvila_decode().k == 12544
    assert synth.llava_next_decode(keep=0.25).k == 720
