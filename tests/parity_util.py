"""Comparison rules shared by the GPU parity tests.

Tolerances (stated once, used everywhere):

* Attention outputs (bf16 out, fp32 accumulation): |gpu - ref| <= 1e-2 +
  2^-8 |ref| elementwise and ||gpu - ref||_2 / ||ref||_2 <= 2e-2, per call.
  The 2^-8 |ref| term is the final round-to-nearest into the bf16 output
  (at least half a bf16 ULP at |ref|): outlier-dominated heads reach |out| ~ 12,
  where one bf16 ULP is 0.0625, so an absolute 1e-2 can only bound the
  arithmetic before that rounding.
* lse (fp32): |gpu - ref| <= 1e-3 (natural-log units).
* Salience (fp32 accumulation of exp over <= 4096 terms, bf16-exact inputs,
  fp32 tensor-core logits): per entry |gpu - ref| / ref <= 1e-4, and every
  row sums to 1 within 1e-5.  Derivation: the logits carry ~1e-7 relative
  error, ex2/lg2 approximations ~2e-7, and fp32 sums of n terms grow the error
  by at most n * 6e-8 (4.4e-5 for n = 729) and typically sqrt(n) * 6e-8.
* Retrieval scores (fp32 GEMV of d <= 128 terms): max |gpu - ref| <=
  1e-5 * max |ref| + 1e-6.
* Softmax-normalised retrieval scores (sums over <= 256 question rows of
  exp(z - lse), fp32 tensor-core logits of bf16 inputs, fp32 lse): per entry
  |gpu - ref| <= 1e-4 |ref| + 1e-7 max|ref|.  The logits carry < 1e-6
  absolute error (fp32 accumulation of d <= 128 exact products of size
  < 64), which is the relative error of each exp; ex2 adds ~2e-7 and the
  row sums ~R*G*6e-8.
* Selected index sets: bit-exact except where scores tie within the band
  delta = 1e-3 * max(|tau|, rms(scores)) around the oracle's k-th score tau;
  the GPU set must have k distinct ascending indices, contain every j with
  s_j > tau + delta and none with s_j < tau - delta.
* Top-k on identical fp32 inputs, compaction, eviction, append: bit-exact.
"""

import numpy as np
import torch

ATTN_ABS = 1e-2
ATTN_REL = 2e-2
BF16_HALF_ULP_REL = 2.0 ** -8
LSE_ABS = 1e-3
SAL_REL = 1e-4
SAL_SUM = 1e-5
SCORE_REL = 1e-5
SOFTMAX_SCORE_REL = 1e-4
TIE_REL = 1e-3


def _f64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().double().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def assert_attention_close(got, ref, what="attention"):
    got = _f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    excess = np.abs(got - ref) - BF16_HALF_ULP_REL * np.abs(ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30)
    i = np.unravel_index(np.argmax(excess), excess.shape)
    assert excess.max() <= ATTN_ABS, (f"{what}: |err| {abs(got[i] - ref[i]):.3g} at |ref| {abs(ref[i]):.3g} "
                                      f"exceeds 1e-2 + 2^-8 |ref|; rel l2 {rel:.3g}")
    assert rel <= ATTN_REL, f"{what}: rel l2 err {rel:.3g} > {ATTN_REL}"


def assert_selection(got, ref_scores, k, what="selection"):
    """got: [..., k] GPU indices; ref_scores: [..., n] oracle fp64 scores."""
    got = np.asarray(got).reshape(-1, k)
    sc = np.asarray(ref_scores, dtype=np.float64).reshape(got.shape[0], -1)
    for row, (g, s) in enumerate(zip(got, sc)):
        assert len(np.unique(g)) == k, f"{what}[{row}]: duplicate indices"
        assert (np.diff(g) > 0).all(), f"{what}[{row}]: not ascending"
        assert g.min() >= 0 and g.max() < len(s), f"{what}[{row}]: index out of range"
        order = np.lexsort((np.arange(len(s)), -s))
        tau = s[order[k - 1]]
        delta = TIE_REL * max(abs(tau), float(np.sqrt(np.mean(s * s))))
        chosen = np.zeros(len(s), bool)
        chosen[g] = True
        missing = np.flatnonzero(~chosen & (s > tau + delta))
        extra = np.flatnonzero(chosen & (s < tau - delta))
        assert missing.size == 0, f"{what}[{row}]: missed {missing[:5]} (tau={tau})"
        assert extra.size == 0, f"{what}[{row}]: wrongly kept {extra[:5]} (tau={tau})"


def assert_salience_close(got, ref, what="salience"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = np.abs(got - ref) / ref
    assert rel.max() <= SAL_REL, f"{what}: max rel err {rel.max():.3g} > {SAL_REL}"
    assert np.abs(got.sum(-1) - 1.0).max() <= SAL_SUM, f"{what}: rows do not sum to 1"


def assert_scores_close(got, ref, what="scores"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref).max()
    bound = SCORE_REL * np.abs(ref).max() + 1e-6
    assert err <= bound, f"{what}: max err {err:.3g} > {bound:.3g}"


def assert_softmax_scores_close(got, ref, what="softmax retrieval scores"):
    got = _f64(got)
    ref = np.asarray(ref, dtype=np.float64)
    bound = SOFTMAX_SCORE_REL * np.abs(ref) + 1e-7 * np.abs(ref).max()
    err = np.abs(got - ref)
    i = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), f"{what}: |err| {err[i]:.3g} at ref {ref[i]:.3g} exceeds the bound {bound[i]:.3g}"
