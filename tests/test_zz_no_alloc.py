"""The workspace-free retrieval entry point, for callers that cannot allocate
device memory (e.g. a plugin inside a framework that owns all device memory,
or a loop where cudaMalloc's possible device synchronisation is forbidden).

It must select exactly what the workspace entry point selects, through the
C ABI, on two calls in a row (the shared fixed scratch keeps the previous
call's contents).  This file is collected last on purpose.
"""

import numpy as np
import pytest
import torch

from visual_token_sparsity_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _cache(shape):
    from visual_token_sparsity_gb300 import binding as sv
    bt = synth.random_block_table(shape.batch, shape.max_blocks, shape.num_blocks, seed=shape.seed + 7)
    lay = synth.draw_decode_layer(shape, 0, bt.to(DEV), device=DEV)
    return sv.KvLayer(lay.k_pool, lay.v_pool), sv.SeqBatch(bt.to(DEV), shape.n_vis, shape.n_text)


@pytest.mark.parametrize("shape", [synth.tiny_decode(batch=2), synth.llava_next_decode(batch=4, keep=0.25, layers=1)],
                         ids=["tiny", "llava-b4"])
def test_noalloc_retrieval_matches_workspace_entry_point(lib, shape):
    from visual_token_sparsity_gb300 import binding as sv
    layer, seqs = _cache(shape)
    B, Hkv, k = shape.batch, shape.Hkv, shape.k
    ws = sv.workspace(sv.sv_retrieve_workspace_bytes(B, shape.H, Hkv, shape.d, shape.n_vis, k))
    for call in range(2):
        qr, _ = synth.draw_decode_queries(shape, 0, device=DEV, step=call)
        ref_idx = torch.empty(B, Hkv, k, dtype=torch.int32, device=DEV)
        ref_sc = torch.empty(B, Hkv, shape.n_vis, device=DEV)
        sv.sv_retrieve_topk(qr, layer, seqs, k, ref_idx, ref_sc, ws)
        idx = torch.full((B, Hkv, k), -1, dtype=torch.int32, device=DEV)
        sc = torch.empty(B, Hkv, shape.n_vis, device=DEV)
        sv.sv_retrieve_topk_noalloc(qr, layer, seqs, k, idx, sc)
        idx2 = torch.full((B, Hkv, k), -1, dtype=torch.int32, device=DEV)
        sv.sv_retrieve_topk_noalloc(qr, layer, seqs, k, idx2)       # scores kept in the fixed scratch
        torch.cuda.synchronize()
        # same kernels, same inputs: identical scores and index sets
        assert torch.equal(sc, ref_sc), f"call {call}: scores differ"
        assert torch.equal(idx, ref_idx), f"call {call}: indices differ"
        assert torch.equal(idx2, ref_idx), f"call {call}: indices (internal scores) differ"


def test_noalloc_rejects_calls_beyond_the_fixed_scratch(lib):
    from visual_token_sparsity_gb300 import binding as sv
    shape = synth.DecodeShape("big", H=8, Hkv=8, d=64, n_vis=262_160, n_text=0, layers=1, batch=1, keep=0.01,
                              seed=5)   # 8 * 262160 scores > 2^21
    bt = torch.zeros(1, shape.max_blocks, dtype=torch.int32, device=DEV)
    pool = torch.zeros(1, 8, 16, 64, dtype=torch.bfloat16, device=DEV)
    layer = sv.KvLayer(pool, pool)
    seqs = sv.SeqBatch(bt, shape.n_vis, 0)
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device=DEV)
    idx = torch.empty(1, 8, 10, dtype=torch.int32, device=DEV)
    with pytest.raises(sv.SvError) as e:
        sv.sv_retrieve_topk_noalloc(q, layer, seqs, 10, idx)
    assert e.value.status == 4 and "scratch" in str(e.value)


def test_noalloc_skips_a_bad_block_like_the_workspace_entry_point(lib):
    """A block-table entry outside the pool: the workspace call reports it in
    its status word; the workspace-free call (whose status word cannot be read
    back) skips the same loads and gives the same indices and scores."""
    from visual_token_sparsity_gb300 import binding as sv
    shape = synth.tiny_decode(batch=2)
    layer, seqs = _cache(shape)
    bt = seqs.block_table.clone()
    bt[1, 3] = shape.num_blocks            # one page of sequence 1 points past the pool
    bad = sv.SeqBatch(bt, shape.n_vis, shape.n_text)
    B, Hkv, k = shape.batch, shape.Hkv, shape.k
    qr, _ = synth.draw_decode_queries(shape, 0, device=DEV)
    ws = sv.workspace(sv.sv_retrieve_workspace_bytes(B, shape.H, Hkv, shape.d, shape.n_vis, k))
    ref_idx = torch.empty(B, Hkv, k, dtype=torch.int32, device=DEV)
    ref_sc = torch.empty(B, Hkv, shape.n_vis, device=DEV)
    sv.sv_retrieve_topk(qr, layer, bad, k, ref_idx, ref_sc, ws)
    assert sv.sv_read_device_status(ws) & sv.SV_DEV_BAD_BLOCK
    idx = torch.full((B, Hkv, k), -1, dtype=torch.int32, device=DEV)
    sc = torch.empty(B, Hkv, shape.n_vis, device=DEV)
    sv.sv_retrieve_topk_noalloc(qr, layer, bad, k, idx, sc)
    torch.cuda.synchronize()
    assert torch.equal(sc, ref_sc)
    assert torch.equal(idx, ref_idx)
    # the skipped page's 16 tokens score 0 in both
    assert (sc[1, :, 48:64] == 0).all()
