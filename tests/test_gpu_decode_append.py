"""GPU: one decode step in one launch (sv_decode_append_attn) against the two
calls it replaces, sv_kv_append of the new token followed by
sv_sparse_decode_attn over the cache that now holds it (velog.io SparseVILA
summary §4.1: a round's answer is decoded token by token, each new token's
K/V entering the cache before it attends).  The outputs, the lse and both
pools must be equal bit for bit, on the CUDA-core kernel (G 1 and 2, both
token steps) and the tensor-core kernel (G 7), with and without an index
list, with per-sequence lengths and with a page outside the pool; one case
is also compared with the oracle."""

import math

import pytest
import torch

import oracle
from parity_util import assert_attention_close
from visual_token_sparsity_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def vis_rows(B, Hkv, n_vis, k, seed):
    g = torch.Generator().manual_seed(seed)
    rows = [torch.sort(torch.randperm(n_vis, generator=g)[:k]).values for _ in range(B * Hkv)]
    return torch.stack(rows).reshape(B, Hkv, k).to(torch.int32).to(DEV)


def setup(H, Hkv, d, n_vis, n_text, B, k, seed):
    """A cache with room for one more token, the step's query and new K/V, and
    two copies of the pools (one per path)."""
    shape = synth.DecodeShape("append", H=H, Hkv=Hkv, d=d, n_vis=n_vis, n_text=n_text, layers=1, batch=B,
                              keep=max(k, 1) / n_vis, seed=seed, extra_blocks=1)
    bt = synth.random_block_table(B, shape.max_blocks, shape.num_blocks, seed=seed + 3).to(DEV)
    lay = synth.draw_decode_layer(shape, 0, bt, device=DEV)
    _, q = synth.draw_decode_queries(shape, 0, device=DEV)
    k_new = synth.normal_bf16((B, Hkv, d), seed + 11, device=DEV)
    v_new = synth.normal_bf16((B, Hkv, d), seed + 12, device=DEV)
    pools = [(lay.k_pool.clone(), lay.v_pool.clone()) for _ in range(2)]
    return shape, bt, q, k_new, v_new, pools


def seq_batch(bt, n_vis, n_text, lens, extra):
    from visual_token_sparsity_gb300 import binding as sv
    if lens is None:
        return sv.SeqBatch(bt, n_vis, n_text + extra)
    nv, nt, ks = lens
    t = lambda xs: torch.tensor(xs, dtype=torch.int32, device=DEV)
    return sv.SeqBatch(bt, n_vis, n_text + extra, t(nv), t([x + extra for x in nt]), t(ks))


def both_paths(shape, bt, q, k_new, v_new, pools, vis, k, lens=None):
    from visual_token_sparsity_gb300 import binding as sv
    B, H, Hkv, d = shape.batch, shape.H, shape.Hkv, shape.d
    scale = 1 / math.sqrt(d)
    n_tok = (k if vis is not None else shape.n_vis) + shape.n_text + 1
    res = []
    for path, (kp, vp) in enumerate(pools):
        layer = sv.KvLayer(kp, vp)
        out = torch.full((B, H, d), 7.0, dtype=torch.bfloat16, device=DEV)
        lse = torch.full((B, H), 7.0, device=DEV)
        ws = sv.workspace(sv.sv_attn_workspace_bytes(B, H, Hkv, d, n_tok))
        if path == 0:
            ws_e = sv.workspace(256)
            sv.sv_kv_append(layer, seq_batch(bt, shape.n_vis, shape.n_text, lens, 0),
                            k_new.view(B, 1, Hkv, d), v_new.view(B, 1, Hkv, d), ws_e)
            sv.sv_sparse_decode_attn(q, scale, layer, seq_batch(bt, shape.n_vis, shape.n_text, lens, 1), vis, k,
                                     out, lse, ws)
            status = sv.sv_read_device_status(ws_e) | sv.sv_read_device_status(ws)
        else:
            sv.sv_decode_append_attn(q, scale, layer, seq_batch(bt, shape.n_vis, shape.n_text, lens, 0), k_new,
                                     v_new, vis, k, out, lse, ws)
            status = sv.sv_read_device_status(ws)
        torch.cuda.synchronize()
        res.append((out, lse, status))
    return res


def assert_same(res, pools):
    (o1, l1, s1), (o2, l2, s2) = res
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)
    assert s1 == s2
    assert torch.equal(pools[0][0], pools[1][0]) and torch.equal(pools[0][1], pools[1][1])


@pytest.mark.parametrize("H,Hkv,d,n_vis,n_text,B,k,indexed", [
    (32, 32, 128, 2880, 128, 4, 1440, True),   # G 1, 8-token steps; the new token is alone in a 29th split
    (4, 2, 64, 576, 32, 1, 144, True),         # the round-loop shape: G 2, 32-token steps
    (28, 4, 128, 3136, 100, 2, 784, True),     # G 7, tensor-core kernel
    (8, 8, 128, 300, 0, 2, 0, False),          # no index list, the new token is the first text token
    (16, 2, 64, 200, 24, 3, 1, True),          # G 8, one visual token, the new token opens a page
    (28, 4, 128, 600, 40, 2, 0, False),        # G 7 without an index list (dense over the cache)
    (8, 8, 64, 500, 10, 1, 100, True),         # 8 units: 32-token steps, G 1, d 64
    (16, 8, 128, 900, 33, 1, 300, True),       # 8 units: 32-token steps, G 2, d 128
])
def test_fused_append_matches_two_calls(lib, H, Hkv, d, n_vis, n_text, B, k, indexed):
    shape, bt, q, k_new, v_new, pools = setup(H, Hkv, d, n_vis, n_text, B, k, seed=H + n_vis + B)
    vis = vis_rows(B, Hkv, n_vis, k, seed=k + 5) if indexed else None
    res = both_paths(shape, bt, q, k_new, v_new, pools, vis, k)
    assert res[0][2] == 0
    assert_same(res, pools)


def test_fused_append_with_per_sequence_lengths(lib):
    nv, nt = [500, 137, 0, 321], [30, 0, 9, 64]
    ks = [250, 60, 0, 321]
    for H, Hkv in ((8, 8), (28, 4)):
        shape, bt, q, k_new, v_new, pools = setup(H, Hkv, 128, max(nv), max(nt), len(nv), max(ks), seed=H + 71)
        vis = vis_rows(len(nv), Hkv, max(nv), max(ks), seed=9)
        # the rows of the index list past each sequence's n_vis are ignored (k_seq <= n_vis_seq)
        vis = torch.where(vis < torch.tensor(nv, device=DEV).view(-1, 1, 1), vis, 0).to(torch.int32)
        vis = torch.sort(vis, dim=-1).values.contiguous()
        res = both_paths(shape, bt, q, k_new, v_new, pools, vis, max(ks), lens=(nv, nt, ks))
        assert res[0][2] == 0
        assert_same(res, pools)


def test_fused_append_with_a_page_outside_the_pool(lib):
    from visual_token_sparsity_gb300 import binding as sv
    shape, bt, q, k_new, v_new, pools = setup(8, 4, 64, 400, 20, 2, 100, seed=33)
    bt[1, (shape.n_vis + shape.n_text) // 16] = shape.num_blocks    # the new token's page of sequence 1
    vis = vis_rows(2, 4, 400, 100, seed=4)
    res = both_paths(shape, bt, q, k_new, v_new, pools, vis, 100)
    assert res[0][2] & sv.SV_DEV_BAD_BLOCK
    assert_same(res, pools)


def test_fused_append_matches_the_oracle(lib):
    shape, bt, q, k_new, v_new, pools = setup(4, 2, 64, 576, 32, 1, 144, seed=5)
    vis = vis_rows(1, 2, 576, 144, seed=6)
    res = both_paths(shape, bt, q, k_new, v_new, pools, vis, 144)
    out = res[1][0]
    # the logical cache after the append: the pages read back through the table
    kp, vp = pools[1]
    n = 576 + 33
    Kl = torch.empty(1, 2, n, 64, dtype=torch.float64)
    Vl = torch.empty_like(Kl)
    btc = bt.cpu()
    for pos in range(n):
        page = int(btc[0, pos // 16])
        Kl[0, :, pos] = kp[page, :, pos % 16].double().cpu()
        Vl[0, :, pos] = vp[page, :, pos % 16].double().cpu()
    # the appended rows are the caller's
    assert torch.equal(Kl[0, :, n - 1], k_new[0].double().cpu())
    o_ref, _ = oracle.sparse_decode_attention(q.double().cpu().numpy(), Kl.numpy(), Vl.numpy(), vis.cpu().numpy(),
                                              576, 33)
    assert_attention_close(out.cpu(), o_ref)


def test_fused_append_replays_in_a_cuda_graph(lib):
    """Captured once and replayed, the fused step gives the eager call's bits
    (no host-side state between calls)."""
    from visual_token_sparsity_gb300 import binding as sv
    shape, bt, q, k_new, v_new, pools = setup(4, 2, 64, 576, 32, 1, 144, seed=41)
    vis = vis_rows(1, 2, 576, 144, seed=42)
    B, H, Hkv, d = 1, 4, 2, 64
    n_tok = 144 + 32 + 1
    outs = []
    for path, (kp, vp) in enumerate(pools):
        layer = sv.KvLayer(kp, vp)
        seqs = sv.SeqBatch(bt, 576, 32)
        out = torch.zeros(B, H, d, dtype=torch.bfloat16, device=DEV)
        ws = sv.workspace(sv.sv_attn_workspace_bytes(B, H, Hkv, d, n_tok))
        call = lambda: sv.sv_decode_append_attn(q, 1 / math.sqrt(d), layer, seqs, k_new, v_new, vis, 144, out,
                                                None, ws)
        if path == 0:
            call()
        else:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                call()
            for _ in range(3):
                g.replay()
        torch.cuda.synchronize()
        assert sv.sv_read_device_status(ws) == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(pools[0][0], pools[1][0]) and torch.equal(pools[0][1], pools[1][1])
