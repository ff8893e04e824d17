"""GPU parity of the prefill salience beyond one SigLIP frame: long sequences
(both operands streamed through 128 x 256 tiles: the QwenVL / video-length
case of the velog.io summary §3.1 kernel paragraph), the head dims of the
other encoders (d 80: Qwen2-VL's vision tower), the boundary between the
resident and the streamed schedule, and inputs whose row sums leave the range
the optimistic first pass accepts, so that the exact re-run is what computes
them.  Each case against oracle.salience on the same bf16 inputs."""

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


def run(q, k, scale=None):
    from visual_token_sparsity_gb300 import binding as sv
    B, H, N, d = q.shape
    sal = torch.empty(B, N, device=DEV)
    ws = sv.workspace(sv.sv_salience_workspace_bytes(B, H, N, d))
    sv.sv_salience_prefill(q.to(DEV), k.to(DEV), scale or 1.0 / math.sqrt(d), sal, ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0
    return sal, ws


def draw(B, H, N, d, seed, std=1.0):
    q = synth.normal_bf16((B, H, N, d), seed, std=std)
    k = synth.normal_bf16((B, H, N, d), seed + 1, std=std)
    synth.scale_token_rows(k, synth.outlier_positions(N, seed + 2), 4.0, token_dim=2)
    return q, k


@pytest.mark.parametrize("N,d", [(4096, 64), (4096, 72), (4096, 80), (4096, 128),
                                 (16384, 64), (16384, 72), (16384, 128)])
def test_long_sequence_salience_matches_oracle(lib, N, d):
    from visual_token_sparsity_gb300 import binding as sv
    assert sv.sv_salience_kernel_count(N, d) == 4      # the streamed schedule
    q, k = draw(1, 1, N, d, seed=N + d)
    sal, _ = run(q, k)
    assert_salience_close(sal.cpu().numpy(), oracle.salience(f64(q), f64(k)), f"N={N} d={d}")


@pytest.mark.parametrize("B,H,N,d", [(1, 2, 1024, 64), (1, 2, 1025, 64), (2, 1, 1300, 72), (1, 2, 768, 80),
                                     (1, 2, 769, 80), (1, 2, 512, 128), (2, 1, 513, 128), (3, 2, 2000, 72),
                                     (1, 3, 257, 80), (2, 2, 33, 80)])
def test_schedule_boundaries_match_oracle(lib, B, H, N, d):
    """Both sides of the resident / streamed switch, ragged tails, d 80."""
    q, k = draw(B, H, N, d, seed=B * 31 + N + d)
    sal, _ = run(q, k)
    assert_salience_close(sal.cpu().numpy(), oracle.salience(f64(q), f64(k)), f"B={B} H={H} N={N} d={d}")


@pytest.mark.parametrize("N,d", [(729, 72), (576, 64), (3000, 72), (700, 128)])
def test_overflowing_row_sums_take_the_exact_path(lib, N, d):
    """Logits of several hundred (log2 units): exp2 of the raw logit
    overflows, so the optimistic row sums are rejected and those heads are
    recomputed with a running max.  One head keeps ordinary logits (mixed
    list).  The result must still match the oracle."""
    q, k = draw(2, 3, N, d, seed=N + 7, std=3.0)
    q[1, 2] = q[1, 2] / 6.0          # ordinary-sized logits for one head
    sal, _ = run(q, k)
    assert np.isfinite(sal.cpu().numpy()).all()
    assert_salience_close(sal.cpu().numpy(), oracle.salience(f64(q), f64(k)), f"N={N} d={d} large logits")


@pytest.mark.parametrize("N,d", [(729, 72), (2500, 64)])
def test_underflowing_row_sums_take_the_exact_path(lib, N, d):
    """Every logit of every row below -140 (log2 units): each exp2 of the raw
    logit flushes to 0 and the optimistic row sum is 0."""
    g = torch.Generator().manual_seed(N)
    u = torch.ones(d)
    noise = lambda: 0.05 * torch.randn(1, 2, N, d, generator=g)
    q = ((3.0 * u) + noise()).to(torch.bfloat16)
    k = ((-2.0 * u) + noise()).to(torch.bfloat16)
    sal, _ = run(q, k)
    assert np.isfinite(sal.cpu().numpy()).all()
    assert_salience_close(sal.cpu().numpy(), oracle.salience(f64(q), f64(k)), f"N={N} d={d} tiny sums")


def test_repeated_calls_reuse_the_failure_list(lib):
    """The exact re-run empties its list: a call with ordinary logits after
    one that needed the re-run, on the same workspace, gives the same bits
    as on a fresh workspace."""
    from visual_token_sparsity_gb300 import binding as sv
    B, H, N, d = 2, 2, 729, 72
    qa, ka = draw(B, H, N, d, seed=5, std=3.0)
    qb, kb = draw(B, H, N, d, seed=9)
    ws = sv.workspace(sv.sv_salience_workspace_bytes(B, H, N, d))
    out = torch.empty(B, N, device=DEV)
    sv.sv_salience_prefill(qa.to(DEV), ka.to(DEV), 1 / math.sqrt(d), out, ws)
    sv.sv_salience_prefill(qb.to(DEV), kb.to(DEV), 1 / math.sqrt(d), out, ws)
    fresh, _ = run(qb, kb)
    assert torch.equal(out, fresh)


def test_long_sequence_deterministic(lib):
    from visual_token_sparsity_gb300 import binding as sv
    q, k = draw(2, 4, 3000, 80, seed=3)
    a, ws = run(q, k)
    b = torch.empty_like(a)
    sv.sv_salience_prefill(q.to(DEV), k.to(DEV), 1 / math.sqrt(80), b, ws)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_long_sequence_zero_queries_exactly_uniform(lib):
    """Q = 0: every logit is 0 and every key is summed in the same order, so
    the salience row is exactly tied (also on the streamed schedule)."""
    N, d = 5000, 72
    q = torch.zeros(1, 2, N, d, dtype=torch.bfloat16)
    k = synth.normal_bf16((1, 2, N, d), 4)
    sal, _ = run(q, k)
    s = sal.cpu().numpy()
    assert (s == s[:, :1]).all()
    assert abs(s[0, 0] - 1.0 / N) <= 1e-7
