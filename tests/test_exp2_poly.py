"""The FMA-pipe exp2 used for part of the forward kernel's exponentials.

The coefficients hard-coded in csrc/fwd_sm103a.cu must be the minimax fit that
exact_attention_tma_gb300/exp2_poly.py reproduces, and the kernel's float32
evaluation (range reduction with the 1.5 * 2^23 rounding trick, Horner,
exponent add) must stay within its error bound against numpy's exp2 -- far
below the 2^-9 relative rounding that P undergoes when it is cast to bf16.
"""
import os
import re

import numpy as np

from exact_attention_tma_gb300.exp2_poly import eval_f32, fit

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "exact_attention_tma_gb300", "csrc", "fwd_sm103a.cu")


def _kernel_coefficients():
    text = open(SRC).read()
    body = text[text.index("float2 exp2_poly2("):]
    body = body[:body.index("return p;")]
    vals = [float(v) for v in re.findall(r"make_float2\(([0-9.e+-]+)f, \1f\)", body)]
    # order in the source: c3, c2, c1, c0 (Horner); skip the rounding constants
    coeffs = [v for v in vals if abs(v) < 2.0 and v != -1.0]
    assert len(coeffs) == 4, coeffs
    return coeffs[::-1]   # ascending: c0..c3


def test_coefficients_are_the_minimax_fit():
    c_src = np.array(_kernel_coefficients())
    c_fit = fit()
    np.testing.assert_allclose(c_src, c_fit, rtol=2e-7, atol=0)


def test_float32_evaluation_error_bound():
    c = _kernel_coefficients()
    x = np.linspace(-30.0, 8.0, 1_000_001).astype(np.float32)
    rel = np.abs(eval_f32(x, c) / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < 1.0e-4
    x = np.linspace(-126.0, -30.0, 200_001).astype(np.float32)
    rel = np.abs(eval_f32(x, c) / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < 2.0e-4


def test_integer_and_half_integer_points():
    c = _kernel_coefficients()
    x = np.arange(-120, 9, 0.5, dtype=np.float32)
    rel = np.abs(eval_f32(x, c) / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < 1.0e-4
