"""Error bound of the FMA-pipe exp2 used by the salience kernel.

The kernel's steps (clamp at -126, round-to-nearest with the 1.5 * 2^23
shifter, degree-4 polynomial on [-1/2, 1/2], exponent added in the integer
domain) are replayed here in float32 with the coefficients read from
csrc/fastmath.cuh, and compared with exp2 in float64."""

import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "visual_token_sparsity_gb300", "csrc", "fastmath.cuh")


def coeffs():
    text = open(SRC).read()
    c = {k: np.float32(float(v)) for k, v in re.findall(r"constexpr float (k\w+) = ([-0-9.e]+)f;", text)}
    return [c[f"kExp2C{i}"] for i in range(5)], c["kShifter"], c["kExp2Min"]


def kernel_exp2(x):
    (c0, c1, c2, c3, c4), shifter, lo = coeffs()
    f32 = np.float32

    def fma(a, b, c):       # single rounding: the fp32 product is exact in fp64
        return (a.astype(np.float64) * b.astype(np.float64) + np.float64(c)).astype(f32)

    xc = np.maximum(x.astype(f32), lo)
    t = (xc + shifter).astype(f32)
    j = (t - shifter).astype(f32)
    f = fma(j, np.full_like(j, -1), xc)
    p = fma(np.full_like(f, c4), f, c3)
    for c in (c2, c1, c0):
        p = fma(p, f, c)
    bits = (p.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << 23)) & 0xFFFFFFFF
    return bits.astype(np.uint32).view(f32)


def test_relative_error_bound_over_the_used_range():
    x = np.linspace(-126.0, 0.0, 2_000_001).astype(np.float32)
    rel = kernel_exp2(x).astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0
    assert np.abs(rel).max() < 3e-6


def test_integer_points_and_clamp():
    x = np.array([0.0, -1.0, -2.0, -10.0, -125.0, -126.0], np.float32)
    np.testing.assert_allclose(kernel_exp2(x), np.exp2(x.astype(np.float64)), rtol=3e-6)
    low = kernel_exp2(np.array([-127.0, -500.0, -np.inf], np.float32))
    assert (low > 0).all() and (low < 2.0 ** -125).all()
