"""GPU parity of the threshold prune (sv_prune_threshold): kept indices,
counts and gathered rows bit-exact against the oracle applied to the same
salience values (the comparison decides the kept set in fp32 on both sides)."""

import math

import numpy as np
import pytest
import torch

import oracle
from visual_token_sparsity_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run(sal, feat, thr):
    from visual_token_sparsity_gb300 import binding as sv
    B, N = sal.shape
    idx = torch.empty(B, N, dtype=torch.int32, device=DEV)
    cnt = torch.empty(B, dtype=torch.int32, device=DEV)
    out = torch.zeros_like(feat) if feat is not None else None
    ws = sv.workspace(sv.sv_prune_workspace_bytes(B, N, 1))
    sv.sv_prune_threshold(sal, thr, feat, out, idx, cnt, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0
    return idx.cpu().numpy(), cnt.cpu().numpy(), None if out is None else out.cpu()


def check(sal, feat, thr):
    idx, cnt, out = run(sal, feat, thr)
    ref = oracle.prune_threshold(sal.cpu().numpy(), feat.cpu().view(torch.int16).numpy(), np.float32(thr))
    for b, (ridx, rrows) in enumerate(ref):
        assert cnt[b] == len(ridx)
        np.testing.assert_array_equal(idx[b, :cnt[b]], ridx)
        assert (idx[b, cnt[b]:] == -1).all()
        np.testing.assert_array_equal(out[b, :cnt[b]].view(torch.int16).numpy(), rrows)


def test_threshold_prune_siglip_mean_salience(lib):
    # keep the above-average tokens of SigLIP-shaped frames (salience from the GPU kernel)
    from visual_token_sparsity_gb300 import binding as sv
    ss = synth.siglip_salience(batch=8)
    q, k, feat = synth.draw_salience(ss, device=DEV)
    sal = torch.empty(ss.batch, ss.N, device=DEV)
    sv.sv_salience_prefill(q, k, 1 / math.sqrt(ss.d), sal,
                           sv.workspace(sv.sv_salience_workspace_bytes(ss.batch, ss.H, ss.N, ss.d)))
    check(sal, feat, 1.0 / ss.N)


@pytest.mark.parametrize("B,N,C,thr", [(3, 1000, 64, 0.0), (2, 7, 16, -math.inf), (2, 7, 16, math.inf),
                                        (1, 5000, 8, 0.5), (4, 33, 256, -0.25)])
def test_threshold_prune_edges(lib, B, N, C, thr):
    g = torch.Generator().manual_seed(B * 1000 + N)
    sal = torch.randn(B, N, generator=g)
    sal[0, ::5] = 0.0                      # ties at a zero threshold: dropped
    feat = synth.normal_bf16((B, N, C), 3).to(DEV)
    check(sal.to(DEV), feat, thr)


def test_threshold_prune_indices_only_and_nan_threshold(lib):
    from visual_token_sparsity_gb300 import binding as sv
    sal = torch.tensor([[0.2, 0.9, -1.0, 0.9]], device=DEV)
    idx, cnt, _ = run(sal, None, 0.5)
    assert cnt[0] == 2 and list(idx[0]) == [1, 3, -1, -1]
    with pytest.raises(RuntimeError):
        run(sal, None, float("nan"))
