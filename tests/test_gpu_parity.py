"""GPU parity: every libsv entry point against the fp64 oracle, through the C ABI.

Small and ragged shapes span several tiles plus a tail; the full workload
shapes are checked on sampled (sequence, head) units the oracle computes one
by one.  Tolerances are documented in parity_util.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import (LSE_ABS, assert_attention_close, assert_salience_close,
                         assert_scores_close, assert_selection)
from visual_token_sparsity_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


def f64(t):
    return t.detach().double().cpu().numpy()


# ------------------------------------------------------------------ top-k

@pytest.mark.parametrize("rows,n,k", [(1, 1, 1), (3, 15, 4), (2, 16, 16), (5, 17, 9), (4, 729, 182),
                                      (7, 2880, 720), (2, 50176, 12544), (1, 60000, 777),
                                      (300, 576, 144), (3, 20000, 1), (2, 40000, 40000), (33, 16385, 4097)])
def test_topk_rows_bit_exact(lib, rows, n, k):
    from visual_token_sparsity_gb300 import binding as sv
    g = torch.Generator().manual_seed(rows * 1000 + n)
    # coarse values force many exact ties; signed zeros included
    x = torch.randint(-40, 40, (rows, n), generator=g).float() / 8.0
    x[x == 0] = -0.0 if n % 2 else 0.0
    x[:, ::7] = torch.randn(rows, (n + 6) // 7, generator=g)
    idx = torch.empty(rows, k, dtype=torch.int32, device=DEV)
    ws = sv.workspace(sv.sv_topk_workspace_bytes(rows, n, k))
    sv.sv_topk_rows(x.to(DEV), k, idx, ws)
    ref = oracle.topk_ascending(x.double().numpy(), k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref)


@pytest.mark.parametrize("n,k", [(20000, 7000), (50176, 12544)])
def test_topk_long_rows_narrow_and_tied(lib, n, k):
    """Long rows (the cluster path): values in a narrow positive range share
    the high key bits (the first radix windows hold one bin), an all-equal
    row takes the lowest indices, and a row of two values straddles k."""
    from visual_token_sparsity_gb300 import binding as sv
    g = torch.Generator().manual_seed(n)
    narrow = 1000.0 + torch.randint(0, 300, (n,), generator=g).float() / 1024.0
    equal = torch.full((n,), -3.5)
    two = torch.where(torch.arange(n) % 3 == 0, torch.tensor(2.0), torch.tensor(1.0))
    x = torch.stack([narrow, equal, two])
    idx = torch.empty(3, k, dtype=torch.int32, device=DEV)
    sv.sv_topk_rows(x.to(DEV), k, idx, sv.workspace(sv.sv_topk_workspace_bytes(3, n, k)))
    np.testing.assert_array_equal(idx.cpu().numpy(), oracle.topk_ascending(x.double().numpy(), k))
    assert (idx.cpu().numpy()[1] == np.arange(k)).all()


def test_topk_all_equal_takes_lowest_indices(lib):
    from visual_token_sparsity_gb300 import binding as sv
    x = torch.full((2, 1000), 0.25, device=DEV)
    idx = torch.empty(2, 300, dtype=torch.int32, device=DEV)
    sv.sv_topk_rows(x, 300, idx, sv.workspace(256))
    assert (idx.cpu().numpy() == np.arange(300)[None]).all()


# ------------------------------------------------------------------ salience

@pytest.mark.parametrize("B,H,N,d,std", [(1, 4, 576, 64, 1.0), (2, 16, 729, 72, 1 / math.sqrt(72)),
                                         (1, 2, 729, 72, 1.0), (3, 1, 1, 64, 1.0), (1, 2, 17, 72, 1.0),
                                         (2, 3, 130, 64, 1.0), (1, 2, 200, 128, 1.0),
                                         (1, 1, 1024, 64, 1.0), (1, 2, 1280, 64, 1.0), (1, 1, 512, 128, 1.0),
                                         (12, 16, 100, 64, 1.0), (20, 16, 257, 72, 1 / math.sqrt(72))])
def test_salience_matches_oracle(lib, B, H, N, d, std):
    from visual_token_sparsity_gb300 import binding as sv
    seed = B * 7 + N
    q = synth.normal_bf16((B, H, N, d), seed, std=std)
    k = synth.normal_bf16((B, H, N, d), seed + 1, std=std)
    synth.scale_token_rows(k, synth.outlier_positions(N, seed + 2), 4.0, token_dim=2)
    sal = torch.empty(B, N, device=DEV)
    ws = sv.workspace(sv.sv_salience_workspace_bytes(B, H, N, d))
    sv.sv_salience_prefill(q.to(DEV), k.to(DEV), 1.0 / math.sqrt(d), sal, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0
    ref = oracle.salience(f64(q), f64(k))
    assert_salience_close(sal.cpu().numpy(), ref)


def test_salience_zero_queries_exactly_uniform_and_prune_takes_first_k(lib):
    from visual_token_sparsity_gb300 import binding as sv
    B, H, N, d = 2, 3, 729, 72
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device=DEV)
    k = synth.normal_bf16((B, H, N, d), 3).to(DEV)
    sal = torch.empty(B, N, device=DEV)
    ws = sv.workspace(sv.sv_salience_workspace_bytes(B, H, N, d))
    sv.sv_salience_prefill(q, k, 1 / math.sqrt(d), sal, ws)
    s = sal.cpu().numpy()
    assert np.abs(s - 1.0 / N).max() <= 1e-7
    # every key sees the same logits (all 0) and the kernel sums them in the
    # same order for every key, so each frame's row is exactly tied ...
    assert (s == s[:, :1]).all(), "Q = 0 salience row is not exactly uniform"
    # ... and a full tie goes to the lowest indices
    kept = torch.empty(B, 182, dtype=torch.int32, device=DEV)
    sv.sv_prune_compact(sal, 182, None, None, kept, ws)
    torch.cuda.synchronize()
    assert (kept.cpu().numpy() == np.arange(182)[None]).all()


@pytest.mark.parametrize("N,k", [(729, 182), (729, 364), (5000, 1250), (1, 1)])
def test_prune_on_exactly_tied_rows_takes_first_k(lib, N, k):
    from visual_token_sparsity_gb300 import binding as sv
    B = 3
    sal = torch.full((B, N), 1.0 / N, device=DEV)
    sal[1] = -0.0      # signed zeros tie with each other
    sal[1, ::2] = 0.0
    ws = sv.workspace(sv.sv_prune_workspace_bytes(B, N, k))
    kept = torch.empty(B, k, dtype=torch.int32, device=DEV)
    sv.sv_prune_compact(sal, k, None, None, kept, ws)
    torch.cuda.synchronize()
    assert (kept.cpu().numpy() == np.arange(k)[None]).all()


def test_salience_deterministic(lib):
    from visual_token_sparsity_gb300 import binding as sv
    B, H, N, d = 4, 16, 729, 72
    q = synth.normal_bf16((B, H, N, d), 11, std=1.0).to(DEV)
    k = synth.normal_bf16((B, H, N, d), 12, std=1.0).to(DEV)
    ws = sv.workspace(sv.sv_salience_workspace_bytes(B, H, N, d))
    a = torch.empty(B, N, device=DEV)
    b = torch.empty(B, N, device=DEV)
    sv.sv_salience_prefill(q, k, 1 / math.sqrt(d), a, ws)
    sv.sv_salience_prefill(q, k, 1 / math.sqrt(d), b, ws)
    assert torch.equal(a, b)


@pytest.mark.parametrize("keep", [0.25, 0.5])
def test_siglip_full_batch_salience_prune_compact_sampled(lib, keep):
    """SigLIP-so400m workload at B = 256 frames; oracle on 3 sampled frames."""
    from visual_token_sparsity_gb300 import binding as sv
    ss = synth.siglip_salience(batch=256, keep=keep)
    q, k, feat = synth.draw_salience(ss, device=DEV)
    sal = torch.empty(ss.batch, ss.N, device=DEV)
    ws = sv.workspace(sv.sv_salience_workspace_bytes(ss.batch, ss.H, ss.N, ss.d))
    sv.sv_salience_prefill(q, k, 1 / math.sqrt(ss.d), sal, ws)
    kept = torch.empty(ss.batch, ss.k, dtype=torch.int32, device=DEV)
    fout = torch.empty(ss.batch, ss.k, ss.C, dtype=torch.bfloat16, device=DEV)
    sv.sv_prune_compact(sal, ss.k, feat, fout, kept, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0
    for b in (0, 131, 255):
        ref = oracle.salience(f64(q[b:b + 1]), f64(k[b:b + 1]))
        assert_salience_close(sal[b:b + 1].cpu().numpy(), ref, f"salience frame {b}")
        assert_selection(kept[b].cpu().numpy(), ref[0], ss.k, f"prune frame {b}")
        kb = kept[b].cpu().long()
        assert torch.equal(fout[b].cpu(), feat[b].cpu()[kb]), "compaction is not a bitwise copy"


def test_prune_compact_bit_exact_on_given_salience(lib):
    from visual_token_sparsity_gb300 import binding as sv
    B, N, k, C = 5, 729, 182, 1152
    g = torch.Generator().manual_seed(9)
    sal = (torch.randint(0, 50, (B, N), generator=g).float() / 1000.0)
    feat = synth.normal_bf16((B, N, C), 10)
    kept = torch.empty(B, k, dtype=torch.int32, device=DEV)
    fout = torch.empty(B, k, C, dtype=torch.bfloat16, device=DEV)
    sv.sv_prune_compact(sal.to(DEV), k, feat.to(DEV), fout, kept, sv.workspace(256))
    idx, out = oracle.prune_compact(sal.double().numpy(), feat.view(torch.int16).numpy(), k)
    np.testing.assert_array_equal(kept.cpu().numpy(), idx)
    np.testing.assert_array_equal(fout.cpu().view(torch.int16).numpy(), out)


# ------------------------------------------------------------------ decode helpers

def make_cache(shape, layer=0, identity=False, device=DEV):
    from visual_token_sparsity_gb300 import binding as sv
    bt = synth.random_block_table(shape.batch, shape.max_blocks, shape.num_blocks,
                                  seed=synth.subseed(shape.seed, layer, 99), identity=identity)
    lay = synth.draw_decode_layer(shape, layer, bt.to(device), device=device)
    return lay, sv.KvLayer(lay.k_pool, lay.v_pool), sv.SeqBatch(bt.to(device), shape.n_vis, shape.n_text)


def random_vis_idx(B, Hkv, n_vis, k, seed, sort=True):
    g = torch.Generator().manual_seed(seed)
    rows = []
    for _ in range(B * Hkv):
        r = torch.randperm(n_vis, generator=g)[:k]
        rows.append(torch.sort(r).values if sort else r)
    return torch.stack(rows).reshape(B, Hkv, k).to(torch.int32)


def run_retrieve(shape, lay, layer, seqs, qr):
    from visual_token_sparsity_gb300 import binding as sv
    B, Hkv = shape.batch, shape.Hkv
    vis = torch.empty(B, Hkv, shape.k, dtype=torch.int32, device=DEV)
    sc = torch.empty(B, Hkv, shape.n_vis, device=DEV)
    ws = sv.workspace(sv.sv_retrieve_workspace_bytes(B, shape.H, Hkv, shape.d, shape.n_vis, shape.k))
    sv.sv_retrieve_topk(qr, layer, seqs, shape.k, vis, sc, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0
    return vis, sc


def run_attn(shape, layer, seqs, qd, vis, k, with_lse=True):
    from visual_token_sparsity_gb300 import binding as sv
    B, H = shape.batch, shape.H
    n_tok = (k if vis is not None else seqs.n_vis) + seqs.n_text
    out = torch.empty(B, H, shape.d, dtype=torch.bfloat16, device=DEV)
    lse = torch.empty(B, H, device=DEV) if with_lse else None
    ws = sv.workspace(sv.sv_attn_workspace_bytes(B, H, shape.Hkv, shape.d, n_tok))
    sv.sv_sparse_decode_attn(qd, 1 / math.sqrt(shape.d), layer, seqs,
                             None if vis is None else vis.to(DEV), k, out, lse, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0
    return out, lse


# ------------------------------------------------------------------ retrieval

@pytest.mark.parametrize("H,Hkv,d,n_vis,n_text,B,R,keep", [
    (4, 2, 64, 576, 32, 1, 1, 0.25),      # tiny decode shape
    (4, 2, 64, 576, 32, 2, 32, 0.25),     # 32 question rows
    (8, 8, 128, 2880, 128, 2, 1, 0.5),    # Llama-2-style MHA, fewer heads
    (28, 4, 128, 4000, 40, 1, 3, 0.3),    # GQA 7 with a ragged visual tail
    (2, 1, 64, 23, 5, 3, 2, 1.0),         # k = n_vis, tiny and ragged
])
def test_retrieve_matches_oracle(lib, H, Hkv, d, n_vis, n_text, B, R, keep):
    shape = synth.DecodeShape("t", H=H, Hkv=Hkv, d=d, n_vis=n_vis, n_text=n_text, layers=1, batch=B,
                              keep=keep, R=R, seed=n_vis + B)
    lay, layer, seqs = make_cache(shape)
    qr, _ = synth.draw_decode_queries(shape, 0, device=DEV)
    vis, sc = run_retrieve(shape, lay, layer, seqs, qr)
    idx_ref, sc_ref = oracle.retrieve_topk(f64(qr), f64(lay.k_logical[:, :, :n_vis]), shape.k)
    assert_scores_close(sc.cpu().numpy(), sc_ref)
    assert_selection(vis.cpu().numpy(), sc_ref, shape.k, "retrieval")


def test_retrieve_rows_equal_presummed_row(lib):
    """Linearity: R rows select what their sum selects."""
    shape = synth.DecodeShape("t", H=4, Hkv=2, d=64, n_vis=576, n_text=32, layers=1, batch=1,
                              keep=0.25, R=32, seed=3)
    lay, layer, seqs = make_cache(shape)
    qr, _ = synth.draw_decode_queries(shape, 0, device=DEV)
    _, sc = run_retrieve(shape, lay, layer, seqs, qr)
    # pre-summed rows, rounded to bf16, change scores only through that rounding
    one = qr.float().sum(dim=1, keepdim=True)
    _, sc_ref = oracle.retrieve_topk(one.double().cpu().numpy(), f64(lay.k_logical[:, :, :576]), shape.k)
    assert_scores_close(sc.cpu().numpy(), sc_ref)


# ------------------------------------------------------------------ attention

@pytest.mark.parametrize("H,Hkv,d,n_vis,n_text,B,k,sort", [
    (4, 2, 64, 576, 32, 1, 144, True),
    (32, 32, 128, 2880, 128, 2, 720, True),
    (32, 32, 128, 2880, 128, 1, 1440, False),
    (28, 4, 128, 6000, 256, 1, 1500, True),
    (8, 1, 128, 100, 3, 2, 37, True),
    (6, 2, 64, 50, 0, 2, 13, True),         # no text tokens
    (6, 2, 64, 50, 7, 2, 1, True),          # a single visual token
    (5, 5, 64, 40, 9, 3, 40, False),        # every visual token, listed unsorted
    (16, 1, 64, 300, 17, 2, 77, True),      # 16 heads per KV head (tensor-core tiles, no padding rows)
    (12, 1, 128, 500, 40, 1, 200, False),   # 12 heads per KV head
    (28, 4, 128, 50176, 256, 1, 12544, True),  # LongVILA shape, one sequence
    (28, 4, 128, 3136, 256, 4, 784, True),     # LongVILA at 16 frames: 32-token splits, merge kernel
    (96, 32, 64, 12000, 100, 2, 9600, True),   # G 3, 64 units: 400-token splits (4 row-id blocks a warp)
    # the CUDA-core kernel steps 32 tokens per warp for at most 8 (sequence,
    # KV head) units and 8 tokens above: both sides of that switch, G 1 and 2
    (8, 8, 128, 2880, 128, 1, 721, True),     # 8 units, G 1
    (9, 9, 128, 2880, 128, 1, 719, False),    # 9 units, G 1
    (8, 4, 64, 1000, 20, 2, 250, True),       # 8 units, G 2
    (16, 8, 128, 2000, 60, 3, 333, True),     # 24 units, G 2
])
def test_sparse_attention_matches_oracle(lib, H, Hkv, d, n_vis, n_text, B, k, sort):
    shape = synth.DecodeShape("t", H=H, Hkv=Hkv, d=d, n_vis=n_vis, n_text=n_text, layers=1, batch=B,
                              keep=k / n_vis, seed=H + n_vis)
    lay, layer, seqs = make_cache(shape)
    _, qd = synth.draw_decode_queries(shape, 0, device=DEV)
    vis = random_vis_idx(B, Hkv, n_vis, k, seed=k + B, sort=sort)
    out, lse = run_attn(shape, layer, seqs, qd, vis, k)
    o_ref, l_ref = oracle.sparse_decode_attention(f64(qd), f64(lay.k_logical), f64(lay.v_logical),
                                                  vis.numpy(), n_vis, n_text)
    assert_attention_close(out, o_ref)
    assert np.abs(lse.cpu().numpy() - l_ref).max() <= LSE_ABS


def test_dense_attention_when_index_list_is_null(lib):
    shape = synth.DecodeShape("t", H=8, Hkv=2, d=128, n_vis=300, n_text=21, layers=1, batch=2, keep=1.0,
                              seed=77)
    lay, layer, seqs = make_cache(shape)
    _, qd = synth.draw_decode_queries(shape, 0, device=DEV)
    out, lse = run_attn(shape, layer, seqs, qd, None, 0)
    o_ref, l_ref = oracle.sparse_decode_attention(f64(qd), f64(lay.k_logical), f64(lay.v_logical),
                                                  None, 300, 21)
    assert_attention_close(out, o_ref)
    # k = n_vis through the index path gives the same numbers
    allidx = torch.arange(300, dtype=torch.int32).expand(2, 2, 300).contiguous()
    out2, _ = run_attn(shape, layer, seqs, qd, allidx, 300)
    assert_attention_close(out2, o_ref)


def test_attention_paging_invariance_bitwise(lib):
    """The same logical cache under two block tables gives identical bits."""
    shape = synth.DecodeShape("t", H=32, Hkv=32, d=128, n_vis=2880, n_text=128, layers=1, batch=2,
                              keep=0.25, seed=1)
    lay_a, layer_a, seqs_a = make_cache(shape, identity=True)
    lay_b, layer_b, seqs_b = make_cache(shape, identity=False)
    assert torch.equal(lay_a.k_logical, lay_b.k_logical)
    _, qd = synth.draw_decode_queries(shape, 0, device=DEV)
    vis = random_vis_idx(2, 32, 2880, 720, seed=1)
    a, _ = run_attn(shape, layer_a, seqs_a, qd, vis, 720)
    b, _ = run_attn(shape, layer_b, seqs_b, qd, vis, 720)
    assert torch.equal(a, b)


def test_bad_block_and_index_set_status_without_fault(lib):
    from visual_token_sparsity_gb300 import binding as sv
    shape = synth.DecodeShape("t", H=4, Hkv=2, d=64, n_vis=64, n_text=8, layers=1, batch=1, keep=0.5,
                              seed=8)
    lay, layer, seqs = make_cache(shape)
    bt = seqs.block_table.clone()
    bt[0, 1] = shape.num_blocks + 5            # out of the pool: flagged and skipped
    bad = sv.SeqBatch(bt, shape.n_vis, shape.n_text)
    _, qd = synth.draw_decode_queries(shape, 0, device=DEV)
    vis = random_vis_idx(1, 2, 64, 32, seed=2)
    vis[0, 0, 0] = 64                           # outside [0, n_vis)
    out = torch.empty(1, 4, 64, dtype=torch.bfloat16, device=DEV)
    ws = sv.workspace(sv.sv_attn_workspace_bytes(1, 4, 2, 64, 40))
    sv.sv_sparse_decode_attn(qd, 0.125, layer, bad, vis.to(DEV), 32, out, None, ws)
    st = sv.sv_read_device_status(ws, clear=True)
    assert st & sv.SV_DEV_BAD_BLOCK and st & sv.SV_DEV_BAD_INDEX
    assert sv.sv_read_device_status(ws) == 0
    # the context is still usable
    good, _ = run_attn(shape, layer, seqs, qd, random_vis_idx(1, 2, 64, 32, seed=2), 32)
    assert torch.isfinite(good.float()).all()


def test_host_rejects_bad_arguments_without_launch(lib):
    from visual_token_sparsity_gb300 import binding as sv
    x = torch.zeros(2, 10, device=DEV)
    idx = torch.empty(2, 11, dtype=torch.int32, device=DEV)
    with pytest.raises(sv.SvError) as e:
        sv.sv_topk_rows(x, 11, idx, sv.workspace(256))
    assert e.value.status == 1
    with pytest.raises(sv.SvError) as e:
        sv.sv_topk_rows(x, 5, idx[:, :5].contiguous(), sv.workspace(16))
    assert e.value.status == 4


# ------------------------------------------------------------------ full workloads (sampled)

@pytest.mark.parametrize("keep", [0.5, 0.25])
@pytest.mark.parametrize("layer_id", [0, 16, 31])
def test_llava_next_full_batch_sampled(lib, keep, layer_id):
    """LLaVA-NeXT-7B decode at B = 16, layers 0, L/2 and L-1: every sequence,
    one KV head each, against the oracle (attention over the GPU's own
    selection, so a tie swap inside the band cannot hide a difference)."""
    shape = synth.llava_next_decode(batch=16, keep=keep)
    lay, layer, seqs = make_cache(shape, layer=layer_id)
    qr, qd = synth.draw_decode_queries(shape, layer_id, device=DEV)
    vis, sc = run_retrieve(shape, lay, layer, seqs, qr)
    out, lse = run_attn(shape, layer, seqs, qd, vis, shape.k)
    rng = np.random.default_rng(int(keep * 100) + layer_id)
    for b, g in zip(range(16), rng.integers(0, 32, 16)):
        kv = f64(lay.k_logical[b:b + 1, g:g + 1])
        _, sc_ref = oracle.retrieve_topk(f64(qr[b:b + 1, :, g:g + 1]), kv[:, :, :shape.n_vis], shape.k)
        assert_scores_close(sc[b, g].cpu().numpy(), sc_ref[0, 0])
        assert_selection(vis[b, g].cpu().numpy(), sc_ref[0, 0], shape.k, f"retrieval b{b} g{g}")
        o_ref, l_ref = oracle.sparse_decode_attention(f64(qd[b:b + 1, g:g + 1]), kv,
                                                      f64(lay.v_logical[b:b + 1, g:g + 1]),
                                                      vis[b:b + 1, g:g + 1].cpu().numpy(),
                                                      shape.n_vis, shape.n_text)
        assert_attention_close(out[b, g], o_ref[0, 0], f"attention b{b} g{g}")
        assert abs(lse[b, g].item() - l_ref[0, 0]) <= LSE_ABS


@pytest.mark.parametrize("layer_id", [0, 14, 27])
def test_longvila_full_batch_sampled(lib, layer_id):
    """LongVILA-7B decode at B = 8, layers 0, L/2 and L-1: every sequence,
    one KV head each (7 query heads), against the oracle over the GPU's own
    selection."""
    shape = synth.longvila_decode(batch=8)
    lay, layer, seqs = make_cache(shape, layer=layer_id)
    qr, qd = synth.draw_decode_queries(shape, layer_id, device=DEV)
    vis, sc = run_retrieve(shape, lay, layer, seqs, qr)
    out, lse = run_attn(shape, layer, seqs, qd, vis, shape.k)
    G = shape.H // shape.Hkv
    for b in range(shape.batch):
        g = (b + layer_id) % shape.Hkv
        kv = f64(lay.k_logical[b:b + 1, g:g + 1])
        _, sc_ref = oracle.retrieve_topk(f64(qr[b:b + 1, :, g * G:(g + 1) * G]), kv[:, :, :shape.n_vis],
                                         shape.k)
        assert_scores_close(sc[b, g].cpu().numpy(), sc_ref[0, 0])
        assert_selection(vis[b, g].cpu().numpy(), sc_ref[0, 0], shape.k, f"retrieval b{b} g{g}")
        o_ref, l_ref = oracle.sparse_decode_attention(f64(qd[b:b + 1, g * G:(g + 1) * G]), kv,
                                                      f64(lay.v_logical[b:b + 1, g:g + 1]),
                                                      vis[b:b + 1, g:g + 1].cpu().numpy(),
                                                      shape.n_vis, shape.n_text)
        assert_attention_close(out[b, g * G:(g + 1) * G], o_ref[0], f"attention b{b} g{g}")
        assert np.abs(lse[b, g * G:(g + 1) * G].cpu().numpy() - l_ref[0]).max() <= LSE_ABS
