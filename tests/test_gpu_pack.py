"""GPU parity of pack-once KV (sv_pack_kv): the packed layer holds exactly
the oracle's gather of the selected visual rows then the text rows, and dense
attention over it returns the same bits as sparse attention over the source
(same tokens, same order, same split plan), within tolerance of the oracle."""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_attention_close
from visual_token_sparsity_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def f64(t):
    return t.detach().double().cpu().numpy()


def logical(pool, bt, n):
    return oracle.paged_view(pool.cpu().view(torch.int16).numpy(), bt.cpu().numpy(), n)


def packed_layer(shape, k, seed):
    """An empty paged layer with room for k + n_text (+ 16 appended) tokens per sequence."""
    from visual_token_sparsity_gb300 import binding as sv
    nblk = synth.blocks_for(k + shape.n_text + 16)
    num_blocks = shape.batch * nblk + 3
    bt = synth.random_block_table(shape.batch, nblk, num_blocks, seed=seed).to(DEV)
    kp = torch.zeros(num_blocks, shape.Hkv, 16, shape.d, dtype=torch.bfloat16, device=DEV)
    vp = torch.zeros_like(kp)
    return sv.KvLayer(kp, vp), sv.SeqBatch(bt, k, shape.n_text)


def random_selection(shape, k, seed):
    g = torch.Generator().manual_seed(seed)
    sel = torch.stack([torch.stack([torch.randperm(shape.n_vis, generator=g)[:k].sort().values
                                    for _ in range(shape.Hkv)]) for _ in range(shape.batch)])
    return sel.to(torch.int32)


@pytest.mark.parametrize("H,Hkv,d,n_vis,n_text,B,k", [
    (4, 2, 64, 576, 32, 1, 144),        # tiny shapes
    (32, 32, 128, 2880, 128, 2, 1440),  # LLaVA-NeXT head layout, 2 sequences
    (28, 4, 128, 3136, 256, 2, 784),    # LongVILA head layout (GQA 7), shortened video
    (8, 2, 64, 100, 0, 3, 37),          # no text tokens
    (8, 8, 128, 40, 9, 2, 40),          # every visual token selected
])
def test_pack_then_dense_equals_sparse(lib, H, Hkv, d, n_vis, n_text, B, k):
    from visual_token_sparsity_gb300 import binding as sv
    shape = synth.DecodeShape("pack", H=H, Hkv=Hkv, d=d, n_vis=n_vis, n_text=n_text, layers=1, batch=B,
                              keep=0.5, seed=41)
    bt = synth.random_block_table(B, shape.max_blocks, shape.num_blocks, seed=synth.subseed(41, 0, 98)).to(DEV)
    lay = synth.draw_decode_layer(shape, 0, bt, device=DEV)
    src, seqs = sv.KvLayer(lay.k_pool, lay.v_pool), sv.SeqBatch(bt, n_vis, n_text)
    vis = random_selection(shape, k, 5).to(DEV)
    dst, dseqs = packed_layer(shape, k, seed=77)
    ws = sv.workspace(256)
    sv.sv_pack_kv(src, seqs, vis, k, dst, dseqs, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0

    n = n_vis + n_text
    Kp, Vp = oracle.pack_selected_kv(logical(lay.k_pool, bt, n), logical(lay.v_pool, bt, n),
                                     vis.cpu().numpy(), n_vis, n_text)
    np.testing.assert_array_equal(logical(dst.k_pool, dseqs.block_table, k + n_text), Kp)
    np.testing.assert_array_equal(logical(dst.v_pool, dseqs.block_table, k + n_text), Vp)

    q = synth.normal_bf16((B, H, d), 9, device=DEV)
    scale = 1.0 / math.sqrt(d)
    wsa = sv.workspace(sv.sv_attn_workspace_bytes(B, H, Hkv, d, k + n_text))
    out_s = torch.empty(B, H, d, dtype=torch.bfloat16, device=DEV)
    out_d = torch.empty_like(out_s)
    lse_s = torch.empty(B, H, device=DEV)
    lse_d = torch.empty_like(lse_s)
    sv.sv_sparse_decode_attn(q, scale, src, seqs, vis, k, out_s, lse_s, wsa)
    sv.sv_sparse_decode_attn(q, scale, dst, dseqs, None, 0, out_d, lse_d, wsa)
    torch.cuda.synchronize()
    assert torch.equal(out_d.view(torch.int16), out_s.view(torch.int16))
    assert torch.equal(lse_d, lse_s)
    ref, ref_lse = oracle.sparse_decode_attention(f64(q), f64(lay.k_logical), f64(lay.v_logical),
                                                  vis.cpu().numpy(), n_vis, n_text, scale)
    assert_attention_close(f64(out_d), ref)
    np.testing.assert_allclose(f64(lse_d), ref_lse, rtol=0, atol=1e-3)


def test_pack_all_visual_and_append_after(lib):
    from visual_token_sparsity_gb300 import binding as sv
    shape = synth.DecodeShape("pack", H=4, Hkv=2, d=64, n_vis=50, n_text=7, layers=1, batch=2, keep=0.5, seed=43)
    bt = synth.random_block_table(2, shape.max_blocks, shape.num_blocks, seed=3).to(DEV)
    lay = synth.draw_decode_layer(shape, 0, bt, device=DEV)
    src, seqs = sv.KvLayer(lay.k_pool, lay.v_pool), sv.SeqBatch(bt, 50, 7)
    dst, dseqs = packed_layer(shape, 50, seed=8)
    ws = sv.workspace(256)
    sv.sv_pack_kv(src, seqs, None, 0, dst, dseqs, ws)
    kn = synth.normal_bf16((2, 3, 2, 64), 1, device=DEV)
    vn = synth.normal_bf16((2, 3, 2, 64), 2, device=DEV)
    sv.sv_kv_append(dst, dseqs, kn, vn, ws)
    torch.cuda.synchronize()
    K2, V2 = oracle.append_tokens(logical(lay.k_pool, bt, 57), logical(lay.v_pool, bt, 57), 57,
                                  kn.cpu().view(torch.int16).numpy(), vn.cpu().view(torch.int16).numpy())
    np.testing.assert_array_equal(logical(dst.k_pool, dseqs.block_table, 60), K2)
    np.testing.assert_array_equal(logical(dst.v_pool, dseqs.block_table, 60), V2)


def test_pack_flags_bad_index_and_rejects_bad_shapes(lib):
    from visual_token_sparsity_gb300 import binding as sv
    shape = synth.DecodeShape("pack", H=4, Hkv=2, d=64, n_vis=40, n_text=4, layers=1, batch=1, keep=0.5, seed=45)
    bt = synth.random_block_table(1, shape.max_blocks, shape.num_blocks, seed=4).to(DEV)
    lay = synth.draw_decode_layer(shape, 0, bt, device=DEV)
    src, seqs = sv.KvLayer(lay.k_pool, lay.v_pool), sv.SeqBatch(bt, 40, 4)
    vis = torch.tensor([[[0, 5, 40], [1, 2, 3]]], dtype=torch.int32, device=DEV)   # 40 is out of range
    dst, dseqs = packed_layer(shape, 3, seed=9)
    ws = sv.workspace(256)
    sv.sv_pack_kv(src, seqs, vis, 3, dst, dseqs, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) & 0x2
    bad = sv.SeqBatch(dseqs.block_table, 2, 4)       # n_vis must equal k
    with pytest.raises(RuntimeError):
        sv.sv_pack_kv(src, seqs, vis, 3, dst, bad, ws)
    with pytest.raises(RuntimeError):                 # packing onto the source pools
        sv.sv_pack_kv(src, seqs, vis, 3, src, dseqs, ws)
