"""GPU parity of the softmax-normalised retrieval (sv_retrieve_topk_softmax)
against the oracle: scores within the stated tolerance, selections exact up
to the tie band, with the normaliser computed here or given by the caller."""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_selection, assert_softmax_scores_close
from visual_token_sparsity_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def f64(t):
    return t.detach().double().cpu().numpy()


def setup(H, Hkv, d, n_vis, n_text, B, R, seed):
    from visual_token_sparsity_gb300 import binding as sv
    shape = synth.DecodeShape("rs", H=H, Hkv=Hkv, d=d, n_vis=n_vis, n_text=n_text, layers=1, batch=B, keep=0.25,
                              seed=seed)
    bt = synth.random_block_table(B, shape.max_blocks, shape.num_blocks, seed=synth.subseed(seed, 0, 98)).to(DEV)
    lay = synth.draw_decode_layer(shape, 0, bt, device=DEV)
    q = synth.normal_bf16((B, R, H, d), seed + 7, device=DEV)
    return lay, sv.KvLayer(lay.k_pool, lay.v_pool), sv.SeqBatch(bt, n_vis, n_text), q


@pytest.mark.parametrize("H,Hkv,d,n_vis,n_text,B,R,k", [
    (4, 2, 64, 576, 64, 1, 32, 144),       # round-loop shapes: 32 question rows
    (32, 32, 128, 2880, 160, 2, 32, 720),  # LLaVA-NeXT head layout
    (28, 4, 128, 3136, 256, 1, 32, 784),   # LongVILA layout: 224 question rows per KV head
    (8, 2, 128, 300, 7, 3, 1, 50),         # one query row
    (16, 1, 64, 1000, 0, 1, 16, 999),      # no text, 256 rows, k = n_vis - 1
])
def test_softmax_retrieval_matches_oracle(lib, H, Hkv, d, n_vis, n_text, B, R, k):
    from visual_token_sparsity_gb300 import binding as sv
    lay, layer, seqs, q = setup(H, Hkv, d, n_vis, n_text, B, R, seed=61)
    scale = 1.0 / math.sqrt(d)
    vis = torch.empty(B, Hkv, k, dtype=torch.int32, device=DEV)
    sc = torch.empty(B, Hkv, n_vis, device=DEV)
    ws = sv.workspace(sv.sv_retrieve_softmax_workspace_bytes(B, R, H, Hkv, d, n_vis, n_text))
    sv.sv_retrieve_topk_softmax(q, scale, layer, seqs, k, vis, sc, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0
    ref = oracle.retrieval_scores_softmax(f64(q), f64(lay.k_logical), n_vis, n_text, scale)
    assert_softmax_scores_close(sc, ref)
    assert_selection(vis.cpu().numpy(), ref, k)


def test_softmax_retrieval_with_given_lse(lib):
    from visual_token_sparsity_gb300 import binding as sv
    B, H, Hkv, d, n_vis, n_text, R, k = 2, 8, 2, 64, 400, 40, 8, 100
    lay, layer, seqs, q = setup(H, Hkv, d, n_vis, n_text, B, R, seed=63)
    scale = 1.0 / math.sqrt(d)
    # a caller's prefill normaliser: here over the visual tokens only
    Kt = lay.k_logical[:, :, :n_vis].double().repeat_interleave(H // Hkv, dim=1)
    lse = torch.logsumexp(torch.einsum("brhd,bhnd->brhn", q.double(), Kt) * scale, dim=-1).float().contiguous()
    vis = torch.empty(B, Hkv, k, dtype=torch.int32, device=DEV)
    sc = torch.empty(B, Hkv, n_vis, device=DEV)
    ws = sv.workspace(sv.sv_retrieve_softmax_workspace_bytes(B, R, H, Hkv, d, n_vis, n_text))
    sv.sv_retrieve_topk_softmax(q, scale, layer, seqs, k, vis, sc, ws, lse=lse)
    torch.cuda.synchronize()
    ref = oracle.retrieval_scores_softmax(f64(q), f64(lay.k_logical), n_vis, n_text, scale, lse=lse.double().cpu().numpy())
    assert_softmax_scores_close(sc, ref)
    np.testing.assert_allclose(f64(sc).sum(-1), R * (H // Hkv), rtol=1e-4)   # visual-only normaliser
    assert_selection(vis.cpu().numpy(), ref, k)


def test_softmax_retrieval_rejects_bad_shapes(lib):
    from visual_token_sparsity_gb300 import binding as sv
    lay, layer, seqs, q = setup(32, 1, 64, 64, 0, 1, 9, seed=65)     # 9 * 32 = 288 rows > 256
    vis = torch.empty(1, 1, 4, dtype=torch.int32, device=DEV)
    ws = sv.workspace(1 << 20)
    with pytest.raises(RuntimeError):
        sv.sv_retrieve_topk_softmax(q, 0.125, layer, seqs, 4, vis, None, ws)
