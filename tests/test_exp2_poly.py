"""The forward kernel's polynomial exp2 (exp2_poly_x2 in fwd_tc.cu), emulated
step by step in float32 on the CPU with the coefficients read from the source.

The kernel clamps x to >= -125, rounds with the 1.5 * 2^23 constant, evaluates
a cubic in f = x - round(x) and adds round(x) into the exponent field.  This
pins the constants and the bit manipulation against the mathematics: 2^x from
float64, exact powers of two at integer x, exactly 1 at x = 0 (a row's max
element gets P = 1 as on the MUFU path), and the stated error bound."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "exact_attention_62_gb300", "csrc", "fwd_tc.cu")


def coefficients():
    text = open(SRC).read()
    return [np.float32(float(re.search(r"constexpr float kExp2C%d = ([0-9.eE+-]+)f;" % i, text).group(1)))
            for i in (1, 2, 3)]


def exp2_poly(x):
    """float32 emulation of the kernel's arithmetic (round-to-nearest, fused
    multiply-add evaluated exactly then rounded, like fma.rn.f32x2)."""
    c1, c2, c3 = coefficients()
    x = np.maximum(np.asarray(x, np.float32), np.float32(-125.0))
    k = np.float32(12582912.0)
    t = (x + k).astype(np.float32)
    j = (t - k).astype(np.float32)
    f = (x.astype(np.float64) - j.astype(np.float64)).astype(np.float32)
    fma = lambda a, b, c: (a.astype(np.float64) * b.astype(np.float64) + np.float64(c)).astype(np.float32)
    q = fma(np.full_like(f, c3), f, c2)
    q = fma(q, f, c1)
    q = fma(q, f, np.float32(1.0))
    bits = (q.view(np.uint32).astype(np.uint64) + (t.view(np.uint32).astype(np.uint64) << np.uint64(23)))
    return (bits & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)


def test_relative_error_bound():
    x = np.concatenate([np.linspace(-125.0, 8.0, 1_000_001, dtype=np.float32),
                        -np.float32(0.5) + np.float32(1e-7) * np.arange(-50, 50, dtype=np.float32)])
    rel = np.abs(exp2_poly(x).astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() <= 1.05e-4, rel.max()


def test_exact_at_integers_and_zero():
    for n in range(-125, 9):
        assert exp2_poly(np.float32(n))[()] == np.float32(2.0) ** n, n
    assert exp2_poly(np.float32(0.0))[()] == np.float32(1.0)
    assert exp2_poly(np.float32(-0.0))[()] == np.float32(1.0)


def test_masked_scores_are_negligible_and_positive():
    y = exp2_poly(np.array([-np.inf, -1e30, -200.0], np.float32))
    assert np.all(y == np.float32(2.0) ** -125)
    # next to a row sum of at least 1 the clamped value vanishes in fp32
    assert np.float32(1.0) + y[0] == np.float32(1.0)


def test_monotone_on_a_fine_grid():
    x = np.linspace(-20.0, 0.0, 400_001, dtype=np.float32)
    y = exp2_poly(x)
    assert np.all(np.diff(y.astype(np.float64)) >= 0)
