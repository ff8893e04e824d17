"""GPU parity of per-sequence lengths (sv_seq_batch n_vis_seq / n_text_seq /
k_seq) through the C ABI.

xllm-io review §五: a threshold prune keeps a different number of visual
tokens per frame, so one decode batch holds sequences with their own visual,
text and selected counts.  Every sequence is compared with the oracle run on
that sequence alone with its own counts.  The cache is filled with random
data up to the capacities, so a kernel that reads past a sequence's own
tokens (or takes its text from the wrong position) changes the result.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import LSE_ABS, assert_attention_close, assert_scores_close, assert_selection
from visual_token_sparsity_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def f64(t):
    return t.detach().double().cpu().numpy()


def varlen_batch(H, Hkv, d, nv, nt, seed, keep=0.5, kseq=None):
    """A cache with capacities max(nv), max(nt) and per-sequence counts."""
    from visual_token_sparsity_gb300 import binding as sv
    B = len(nv)
    shape = synth.DecodeShape("varlen", H=H, Hkv=Hkv, d=d, n_vis=max(nv), n_text=max(nt), layers=1,
                              batch=B, keep=keep, seed=seed, extra_blocks=1)
    bt = synth.random_block_table(B, shape.max_blocks, shape.num_blocks, seed=seed + 5).to(DEV)
    lay = synth.draw_decode_layer(shape, 0, bt, device=DEV)
    if kseq is None:
        kseq = [int(math.floor(keep * n)) for n in nv]
    t = lambda xs: torch.tensor(xs, dtype=torch.int32, device=DEV)
    seqs = sv.SeqBatch(bt, shape.n_vis, shape.n_text, t(nv), t(nt), t(kseq))
    return shape, lay, sv.KvLayer(lay.k_pool, lay.v_pool), seqs, kseq


def retrieve(shape, layer, seqs, qr, k_cap, noalloc=False):
    from visual_token_sparsity_gb300 import binding as sv
    B, Hkv = shape.batch, shape.Hkv
    vis = torch.full((B, Hkv, k_cap), 12345, dtype=torch.int32, device=DEV)
    sc = torch.full((B, Hkv, shape.n_vis), 7.0, device=DEV)
    if noalloc:
        sv.sv_retrieve_topk_noalloc(qr, layer, seqs, k_cap, vis, sc)
        torch.cuda.synchronize()
        return vis, sc, 0
    ws = sv.workspace(sv.sv_retrieve_workspace_bytes(B, shape.H, Hkv, shape.d, shape.n_vis, k_cap))
    sv.sv_retrieve_topk(qr, layer, seqs, k_cap, vis, sc, ws)
    torch.cuda.synchronize()
    return vis, sc, sv.sv_read_device_status(ws)


def attend(shape, layer, seqs, qd, vis, k_cap):
    from visual_token_sparsity_gb300 import binding as sv
    B, H = shape.batch, shape.H
    n_tok = (k_cap if vis is not None else shape.n_vis) + shape.n_text
    out = torch.full((B, H, shape.d), 3.0, dtype=torch.bfloat16, device=DEV)
    lse = torch.full((B, H), 5.0, device=DEV)
    ws = sv.workspace(sv.sv_attn_workspace_bytes(B, H, shape.Hkv, shape.d, n_tok))
    sv.sv_sparse_decode_attn(qd, 1 / math.sqrt(shape.d), layer, seqs, vis, k_cap, out, lse, ws)
    torch.cuda.synchronize()
    return out, lse, sv.sv_read_device_status(ws)


def check_retrieval(shape, lay, qr, vis, sc, nv, kseq, k_cap, valid=None):
    K = f64(lay.k_logical)
    for b in range(shape.batch):
        row = vis[b].cpu().numpy()
        if valid is not None and not valid[b]:
            assert (row == -1).all(), f"sequence {b}: skipped rows must read -1"
            continue
        kb = kseq[b]
        assert (row[:, kb:] == -1).all(), f"sequence {b}: slots past k_seq must read -1"
        if kb == 0:
            continue
        _, ref = oracle.retrieve_topk(f64(qr[b:b + 1]), K[b:b + 1, :, :nv[b]], kb)
        assert_scores_close(sc[b:b + 1, :, :nv[b]].cpu().numpy(), ref)
        assert_selection(row[None, :, :kb], ref, kb, f"retrieval sequence {b}")
        # entries past the sequence's own visual tokens are left as they were
        assert (sc[b, :, nv[b]:] == 7.0).all()


def check_attention(shape, lay, qd, vis, out, lse, nv, nt, kseq, valid=None):
    K, V = f64(lay.k_logical), f64(lay.v_logical)
    for b in range(shape.batch):
        if (valid is not None and not valid[b]) or (nv[b] if vis is None else kseq[b]) + nt[b] == 0:
            assert (out[b].float() == 0).all(), f"sequence {b}: nothing attended, output must be 0"
            assert torch.isinf(lse[b]).all() and (lse[b] < 0).all()
            continue
        sel = None if vis is None else vis[b:b + 1, :, :kseq[b]].cpu().numpy()
        o_ref, l_ref = oracle.sparse_decode_attention(f64(qd[b:b + 1]), K[b:b + 1], V[b:b + 1], sel,
                                                      nv[b], nt[b])
        assert_attention_close(out[b:b + 1], o_ref, f"attention sequence {b}")
        assert np.abs(lse[b:b + 1].cpu().numpy() - l_ref).max() <= LSE_ABS


@pytest.mark.parametrize("H,Hkv,d,nv,nt,kseq", [
    # G = 1 (CUDA-core attention, fused top-k): full, ragged, one token, k = n_vis, no text, k = 0
    (4, 4, 128, [300, 257, 1, 190, 64, 120], [40, 3, 17, 0, 25, 40], [150, 128, 1, 190, 32, 0]),
    # G = 2, d = 64; a sequence with neither visual nor text tokens
    (8, 4, 64, [200, 0, 77, 199], [9, 0, 31, 1], None),
    # G = 7 (tensor-core attention); a text-only sequence
    (28, 4, 128, [700, 333, 0, 512], [256, 100, 60, 0], None),
])
def test_varlen_retrieve_and_attend(lib, H, Hkv, d, nv, nt, kseq):
    shape, lay, layer, seqs, kseq = varlen_batch(H, Hkv, d, nv, nt, seed=sum(nv) + H, kseq=kseq)
    k_cap = max(1, max(kseq))
    qr, qd = synth.draw_decode_queries(shape, 0, device=DEV)
    vis, sc, st = retrieve(shape, layer, seqs, qr, k_cap)
    assert st == 0
    check_retrieval(shape, lay, qr, vis, sc, nv, kseq, k_cap)
    out, lse, st = attend(shape, layer, seqs, qd, vis, k_cap)
    assert st == 0
    check_attention(shape, lay, qd, vis, out, lse, nv, nt, kseq)
    # dense attention (no index list): every visual token of each sequence
    out, lse, st = attend(shape, layer, seqs, qd, None, 0)
    assert st == 0
    check_attention(shape, lay, qd, None, out, lse, nv, nt, kseq)


@pytest.mark.parametrize("n_cap", [14000, 20000])
def test_varlen_long_rows_standalone_topk(lib, n_cap):
    """Rows too long for the fused top-k: the one-CTA (14000) and the cluster
    (20000) row top-k read the per-sequence counts; the workspace-free entry
    point shares them."""
    nv, nt = [n_cap, n_cap - 2345, 5000], [16, 0, 7]
    kseq = [n_cap // 4, 0, 4999]
    shape, lay, layer, seqs, kseq = varlen_batch(8, 2, 64, nv, nt, seed=n_cap, kseq=kseq)
    qr, _ = synth.draw_decode_queries(shape, 0, device=DEV)
    k_cap = max(kseq)
    vis, sc, st = retrieve(shape, layer, seqs, qr, k_cap)
    assert st == 0
    check_retrieval(shape, lay, qr, vis, sc, nv, kseq, k_cap)
    vis2, _, _ = retrieve(shape, layer, seqs, qr, k_cap, noalloc=True)
    assert torch.equal(vis, vis2)


def test_uniform_lengths_through_arrays_match_the_scalars(lib):
    """Per-sequence arrays that repeat the batch-wide counts give the same bits."""
    from visual_token_sparsity_gb300 import binding as sv
    nv, nt = [576] * 3, [32] * 3
    shape, lay, layer, seqs, kseq = varlen_batch(4, 2, 64, nv, nt, seed=11, keep=0.25)
    plain = sv.SeqBatch(seqs.block_table, shape.n_vis, shape.n_text)
    qr, qd = synth.draw_decode_queries(shape, 0, device=DEV)
    v1, s1, _ = retrieve(shape, layer, seqs, qr, 144)
    v2, s2, _ = retrieve(shape, layer, plain, qr, 144)
    assert torch.equal(v1, v2) and torch.equal(s1, s2)
    o1, l1, _ = attend(shape, layer, seqs, qd, v1, 144)
    o2, l2, _ = attend(shape, layer, plain, qd, v2, 144)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_varlen_append_writes_after_each_sequence(lib):
    from visual_token_sparsity_gb300 import binding as sv
    nv, nt = [100, 37, 64], [5, 0, 20]
    shape, lay, layer, seqs, _ = varlen_batch(4, 2, 64, nv, nt, seed=21)
    T = 3
    kn = synth.normal_bf16((shape.batch, T, shape.Hkv, shape.d), 31, device=DEV)
    vn = synth.normal_bf16((shape.batch, T, shape.Hkv, shape.d), 32, device=DEV)
    before_k, before_v = lay.k_pool.clone(), lay.v_pool.clone()
    ws = sv.workspace(sv.sv_evict_workspace_bytes())
    sv.sv_kv_append(layer, seqs, kn, vn, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0
    bt = seqs.block_table.cpu().numpy()
    touched = torch.zeros(lay.k_pool.shape[:3], dtype=torch.bool)
    for b in range(shape.batch):
        for t in range(T):
            pos = nv[b] + nt[b] + t
            blk, row = bt[b, pos // 16], pos % 16
            assert torch.equal(lay.k_pool[blk, :, row].cpu(), kn[b, t].cpu())
            assert torch.equal(lay.v_pool[blk, :, row].cpu(), vn[b, t].cpu())
            touched[blk, :, row] = True
    assert torch.equal(lay.k_pool.cpu()[~touched], before_k.cpu()[~touched]), "append wrote elsewhere"
    assert torch.equal(lay.v_pool.cpu()[~touched], before_v.cpu()[~touched]), "append wrote elsewhere"


def test_out_of_range_lengths_are_reported_and_skipped(lib):
    from visual_token_sparsity_gb300 import binding as sv
    nv, nt = [200, 150, 90], [10, 10, 10]
    kseq = [100, 151, 45]             # sequence 1 selects more than it has
    shape, lay, layer, seqs, kseq = varlen_batch(4, 2, 64, nv, nt, seed=41, kseq=kseq)
    qr, qd = synth.draw_decode_queries(shape, 0, device=DEV)
    k_cap = 151
    vis, sc, st = retrieve(shape, layer, seqs, qr, k_cap)
    assert st == sv.SV_DEV_BAD_LENGTH
    valid = [True, False, True]
    check_retrieval(shape, lay, qr, vis, sc, nv, kseq, k_cap, valid=valid)
    vis[1] = 0                        # any in-range list: the lengths alone reject sequence 1
    out, lse, st = attend(shape, layer, seqs, qd, vis, k_cap)
    assert st == sv.SV_DEV_BAD_LENGTH
    check_attention(shape, lay, qd, vis, out, lse, nv, nt, kseq, valid=valid)
    # a text count above the capacity
    bad = sv.SeqBatch(seqs.block_table, shape.n_vis, shape.n_text, seqs.n_vis_seq,
                      torch.tensor([10, 11, 10], dtype=torch.int32, device=DEV), None)
    out, lse, st = attend(shape, layer, bad, qd, None, 0)
    assert st == sv.SV_DEV_BAD_LENGTH
    check_attention(shape, lay, qd, None, out, lse, nv, nt, kseq, valid=valid)


def test_calls_without_per_sequence_support_reject_the_arrays(lib):
    from visual_token_sparsity_gb300 import binding as sv
    shape, lay, layer, seqs, _ = varlen_batch(4, 2, 64, [64, 32], [8, 8], seed=51)
    qr, _ = synth.draw_decode_queries(shape, 0, device=DEV, rows=2)
    ws = sv.workspace(1 << 20)
    vis = torch.zeros(shape.batch, shape.Hkv, 16, dtype=torch.int32, device=DEV)
    with pytest.raises(sv.SvError) as e:
        sv.sv_retrieve_topk_softmax(qr, 0.125, layer, seqs, 16, vis, None, ws)
    assert e.value.status == 2
    with pytest.raises(sv.SvError) as e:
        sv.sv_evict_qa_tokens([layer], seqs, 0, 4, ws)
    assert e.value.status == 2
    dst = sv.KvLayer(torch.zeros_like(lay.k_pool), torch.zeros_like(lay.v_pool))
    dseqs = sv.SeqBatch(seqs.block_table, 16, shape.n_text)
    with pytest.raises(sv.SvError) as e:
        sv.sv_pack_kv(layer, seqs, vis, 16, dst, dseqs, ws)
    assert e.value.status == 2


def test_binding_checks_the_per_sequence_arrays(lib):
    from visual_token_sparsity_gb300 import binding as sv
    bt = torch.zeros(3, 4, dtype=torch.int32, device=DEV)
    nv = torch.tensor([40, 10, 0], dtype=torch.int32, device=DEV)
    s = sv.SeqBatch(bt, 40, 8, nv, None, nv)
    assert s.c.n_vis_seq == nv.data_ptr() and s.c.k_seq == nv.data_ptr() and not s.c.n_text_seq
    with pytest.raises(ValueError):
        sv.SeqBatch(bt, 40, 8, torch.zeros(2, dtype=torch.int32, device=DEV))
    with pytest.raises(ValueError):
        sv.SeqBatch(bt, 40, 8, None, torch.zeros(3, dtype=torch.int64, device=DEV))
