"""Programmatic dependent launch changes when a kernel's CTAs become
resident, never what they compute: the decode path (retrieval + sparse
attention over several layers, many rows and a few rows, G 1 and G 7) and the
prefill path (salience, top-k prune + compaction, threshold prune, summary
salience) give the same bits with it on (the default) and off (SV_PDL=0, in a
child process, since the library reads the switch once)."""

import os
import subprocess
import sys
import textwrap

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RUN = textwrap.dedent("""
    import math, sys, torch
    sys.path.insert(0, {root!r})
    from visual_token_sparsity_gb300 import binding as sv, synth
    out = {{}}
    for name, shape in (("mha_b6", synth.DecodeShape("t", H=8, Hkv=8, d=128, n_vis=2880, n_text=64,
                                                      layers=3, batch=10, keep=0.25, seed=5)),
                        ("mha_b1", synth.DecodeShape("t", H=8, Hkv=8, d=128, n_vis=700, n_text=9,
                                                      layers=3, batch=1, keep=0.5, seed=6)),
                        ("gqa", synth.DecodeShape("t", H=28, Hkv=4, d=128, n_vis=20000, n_text=40,
                                                  layers=2, batch=2, keep=0.25, seed=7))):
        bt = synth.random_block_table(shape.batch, shape.max_blocks, shape.num_blocks, seed=3).cuda()
        seqs = sv.SeqBatch(bt, shape.n_vis, shape.n_text)
        ws_r = sv.workspace(sv.sv_retrieve_workspace_bytes(shape.batch, shape.H, shape.Hkv, shape.d,
                                                           shape.n_vis, shape.k))
        ws_a = sv.workspace(sv.sv_attn_workspace_bytes(shape.batch, shape.H, shape.Hkv, shape.d,
                                                       shape.k + shape.n_text))
        for l in range(shape.layers):
            lay = synth.draw_decode_layer(shape, l, bt, device="cuda")
            layer = sv.KvLayer(lay.k_pool, lay.v_pool)
            qr, qd = synth.draw_decode_queries(shape, l, device="cuda")
            vis = torch.empty(shape.batch, shape.Hkv, shape.k, dtype=torch.int32, device="cuda")
            o = torch.empty(shape.batch, shape.H, shape.d, dtype=torch.bfloat16, device="cuda")
            sv.sv_retrieve_topk(qr, layer, seqs, shape.k, vis, None, ws_r)
            sv.sv_sparse_decode_attn(qd, 1 / math.sqrt(shape.d), layer, seqs, vis, shape.k, o, None, ws_a)
            out[f"{{name}}_vis{{l}}"] = vis.cpu()
            out[f"{{name}}_out{{l}}"] = o.cpu()
    ss = synth.siglip_salience(batch=8)
    q, k, feat = synth.draw_salience(ss, device="cuda")
    sal = torch.empty(ss.batch, ss.N, device="cuda")
    ws = sv.workspace(sv.sv_salience_workspace_bytes(ss.batch, ss.H, ss.N, ss.d))
    sv.sv_salience_prefill(q, k, 1 / math.sqrt(ss.d), sal, ws)
    kept = torch.empty(ss.batch, ss.k, dtype=torch.int32, device="cuda")
    fout = torch.empty(ss.batch, ss.k, ss.C, dtype=torch.bfloat16, device="cuda")
    sv.sv_prune_compact(sal, ss.k, feat, fout, kept, ws)
    tidx = torch.empty(ss.batch, ss.N, dtype=torch.int32, device="cuda")
    tcnt = torch.empty(ss.batch, dtype=torch.int32, device="cuda")
    tout = torch.empty(ss.batch, ss.N, ss.C, dtype=torch.bfloat16, device="cuda")
    sv.sv_prune_threshold(sal, 1.0 / ss.N, feat, tout, tidx, tcnt, ws)
    cs = synth.clip_summary_salience(batch=4)
    cq, ck, _ = synth.draw_salience(cs, device="cuda")
    csal = torch.empty(cs.batch, cs.N, device="cuda")
    sv.sv_salience_summary(cq, ck, 1, 1 / math.sqrt(cs.d), csal,
                           sv.workspace(sv.sv_salience_summary_workspace_bytes(cs.batch, cs.H, cs.N, cs.d, 1)))
    for key, t in (("sal", sal), ("kept", kept), ("fout", fout), ("tidx", tidx), ("tcnt", tcnt),
                   ("tout", tout), ("csal", csal)):
        out[key] = t.cpu()
    torch.cuda.synchronize()
    torch.save(out, sys.argv[1])
""")


def run(path, pdl):
    env = dict(os.environ)
    env["SV_PDL"] = "1" if pdl else "0"
    script = RUN.format(root=ROOT)
    r = subprocess.run([sys.executable, "-c", script, path], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    return torch.load(path)


def test_programmatic_launch_does_not_change_results(lib, tmp_path):
    on = run(str(tmp_path / "on.pt"), True)
    off = run(str(tmp_path / "off.pt"), False)
    assert on.keys() == off.keys()
    for key in on:
        if key == "tout":   # rows past a frame's kept count are not written
            continue
        assert torch.equal(on[key], off[key]), key
    for b, n in enumerate(on["tcnt"].tolist()):
        assert torch.equal(on["tout"][b, :n], off["tout"][b, :n]), b
