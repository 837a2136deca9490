"""Fit of the polynomial the forward kernel uses for part of its exp2 calls.

Method: Cody-Waite style range reduction, 2^x = 2^j * 2^f with j = round(x)
and f = x - j in [-1/2, 1/2], then a degree-3 polynomial for 2^f whose maximum
relative error on [-1/2, 1/2] is minimised (minimax) by Lawson's iteratively
reweighted least-squares algorithm on a dense grid.  The kernel rounds with
the float32 "add 1.5 * 2^23" trick and adds j to the exponent field.

Run ``python -m exact_attention_tma_gb300.exp2_poly`` to print the
coefficients that csrc/fwd_sm103a.cu hard-codes; tests/test_exp2_poly.py
re-fits them and checks the float32 evaluation against numpy's exp2.
"""
from __future__ import annotations

import numpy as np


def fit(degree: int = 3, iters: int = 200, grid: int = 20001) -> np.ndarray:
    """Coefficients c[0..degree] (ascending powers) minimising max |p(f)/2^f - 1|."""
    f = np.linspace(-0.5, 0.5, grid)
    y = np.exp2(f)
    A = np.vander(f, degree + 1, increasing=True) / y[:, None]   # relative-error system
    w = np.full(grid, 1.0 / grid)
    c = None
    for _ in range(iters):
        sw = np.sqrt(w)
        c, *_ = np.linalg.lstsq(A * sw[:, None], sw, rcond=None)
        err = np.abs(A @ c - 1.0)
        w = w * err
        w /= w.sum()
    return c


def eval_f32(x: np.ndarray, c) -> np.ndarray:
    """The kernel's float32 evaluation of 2^x for x >= -126, step by step."""
    x = np.asarray(x, dtype=np.float32)
    magic = np.float32(12582912.0)            # 1.5 * 2^23
    t = (x + magic).astype(np.float32)        # round(x) lands in the low mantissa bits
    j = (t - magic).astype(np.float32)
    f = (x - j).astype(np.float32)
    c = [np.float32(v) for v in c]
    p = np.float32(c[3])
    p = (p * f + c[2]).astype(np.float32)
    p = (p * f + c[1]).astype(np.float32)
    p = (p * f + c[0]).astype(np.float32)
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.astype(np.uint32).view(np.float32)


if __name__ == "__main__":
    coef = fit()
    f = np.linspace(-0.5, 0.5, 200001)
    rel = np.abs(np.polyval(coef[::-1], f) / np.exp2(f) - 1).max()
    print("coefficients (c0..c3):", ", ".join(f"{v:.9e}" for v in coef))
    print(f"max relative error on [-1/2, 1/2]: {rel:.3e}")
