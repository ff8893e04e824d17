"""GPU parity of the summary-row salience (CLIP / RADIO rows of the encoder
table) against the oracle, plus its reduction to the full salience."""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_util import assert_salience_close
from visual_token_sparsity_gb300 import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def f64(t):
    return t.detach().double().cpu().numpy()


@pytest.mark.parametrize("B,H,N,d,R,std", [
    (2, 16, 577, 64, 1, 1 / 8),      # CLIP ViT-L/14-336: CLS + 24 x 24 patches
    (1, 16, 1029, 80, 5, 1.0),       # RADIO-like: 5 summary tokens, d 80
    (3, 4, 200, 72, 3, 1.0),
    (1, 2, 5, 64, 5, 1.0),           # every token a summary token
    (2, 1, 1, 128, 1, 1.0),          # a single token
    (1, 3, 2000, 128, 16, 1.0),      # largest R
    (1, 2, 33, 256, 2, 1.0),         # largest head dim
    (2, 9, 150, 64, 1, 1.0),         # an odd head count
    (1, 20, 300, 64, 2, 1.0),        # 20 heads
])
def test_summary_salience_matches_oracle(lib, B, H, N, d, R, std):
    from visual_token_sparsity_gb300 import binding as sv
    seed = 100 + N + R
    q = synth.normal_bf16((B, H, N, d), seed, std=std)
    k = synth.normal_bf16((B, H, N, d), seed + 1, std=std)
    synth.scale_token_rows(k, synth.outlier_positions(N, seed + 2), 4.0, token_dim=2)
    sal = torch.empty(B, N, device=DEV)
    ws = sv.workspace(sv.sv_salience_summary_workspace_bytes(B, H, N, d, R))
    sv.sv_salience_summary(q.to(DEV), k.to(DEV), R, 1.0 / math.sqrt(d), sal, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0
    assert_salience_close(sal.cpu().numpy(), oracle.summary_salience(f64(q), f64(k), R))


def test_summary_salience_deterministic(lib):
    from visual_token_sparsity_gb300 import binding as sv
    B, H, N, d = 4, 16, 577, 64
    q = synth.normal_bf16((B, H, N, d), 21, std=1 / 8).to(DEV)
    k = synth.normal_bf16((B, H, N, d), 22, std=1 / 8).to(DEV)
    ws = sv.workspace(sv.sv_salience_summary_workspace_bytes(B, H, N, d, 1))
    a = torch.empty(B, N, device=DEV)
    b = torch.empty(B, N, device=DEV)
    sv.sv_salience_summary(q, k, 1, 0.125, a, ws)
    sv.sv_salience_summary(q, k, 1, 0.125, b, ws)
    assert torch.equal(a, b)


def test_summary_salience_with_all_rows_equals_full_salience(lib):
    from visual_token_sparsity_gb300 import binding as sv
    B, H, N, d = 1, 4, 12, 64
    q = synth.normal_bf16((B, H, N, d), 7).to(DEV)
    k = synth.normal_bf16((B, H, N, d), 8).to(DEV)
    a = torch.empty(B, N, device=DEV)
    b = torch.empty(B, N, device=DEV)
    sv.sv_salience_summary(q, k, N, 0.125, a, sv.workspace(sv.sv_salience_summary_workspace_bytes(B, H, N, d, N)))
    sv.sv_salience_prefill(q, k, 0.125, b, sv.workspace(sv.sv_salience_workspace_bytes(B, H, N, d)))
    torch.cuda.synchronize()
    np.testing.assert_allclose(a.cpu().numpy(), b.cpu().numpy(), rtol=2e-4, atol=0)


def test_summary_salience_rejects_bad_shapes(lib):
    from visual_token_sparsity_gb300 import binding as sv
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16, device=DEV)
    sal = torch.empty(1, 8, device=DEV)
    ws = sv.workspace(1 << 16)
    for R in (0, 9, 17):
        with pytest.raises(RuntimeError):
            sv.sv_salience_summary(q, q, R, 0.1, sal, ws)
    q60 = torch.zeros(1, 2, 8, 60, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(RuntimeError):
        sv.sv_salience_summary(q60, q60, 1, 0.1, sal, ws)
