"""Parity helpers shared by the GPU tests: run the fp64 oracle on the same
bf16 inputs the kernels saw and compare element by element.

Tolerances (absolute, over all compared elements): bf16 O within
max |err| <= 1.5e-2 and mean |err| <= 2e-3 of the fp64 result; fp32 LSE
within 1e-3.  They cover bf16 rounding of P before the P V product, the
final bf16 rounding of O (half an ulp, <= 7.8e-3 for |O| < 4) and fp32
accumulation order.
"""
import numpy as np
import torch

import oracle

O_MAX, O_MEAN, LSE_MAX = 1.5e-2, 2e-3, 1e-3


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def oracle_fwd(q, k, v, scale, causal, heads=None, rows=None, threads=None):
    """Oracle O, LSE for flat head indices ``heads`` (default all) and query
    ``rows`` (default all).  Returns arrays shaped (nheads, nrows, d)/(nheads, nrows)."""
    B, H, N, d = q.shape
    hs = list(range(B * H)) if heads is None else list(heads)
    qf = q.reshape(B * H, N, d)
    kf = k.reshape(B * H, N, d)
    vf = v.reshape(B * H, N, d)
    Q = to_f64(qf[hs])
    K = to_f64(kf[hs])
    V = to_f64(vf[hs])
    O, LSE = oracle.attention(Q, K, V, scale, causal, rows=rows, threads=threads)
    return O, LSE


def oracle_fwd_head_rows(q, k, v, scale, causal, head, rows, threads=None):
    """Oracle O, LSE of one flat head at the given query rows, the rows split
    over host threads (rows are independent; each chunk is one oracle call).
    Returns arrays shaped (1, len(rows), d) / (1, len(rows))."""
    from concurrent.futures import ThreadPoolExecutor
    import os

    rows = list(rows)
    threads = threads or min(len(rows), os.cpu_count() or 1)
    chunks = [rows[i::threads] for i in range(threads)]
    B, H, N, d = q.shape
    Q = to_f64(q.reshape(B * H, N, d)[head:head + 1])
    K = to_f64(k.reshape(-1, N, d)[head:head + 1])
    V = to_f64(v.reshape(-1, N, d)[head:head + 1])
    with ThreadPoolExecutor(max_workers=threads) as ex:
        parts = list(ex.map(lambda c: oracle.attention(Q, K, V, scale, causal, rows=c, threads=1),
                            chunks))
    O = np.empty((1, len(rows), d))
    L = np.empty((1, len(rows)))
    for i, (o, l) in enumerate(parts):
        O[0, i::threads] = o[0]
        L[0, i::threads] = l[0]
    return O, L


def compare_fwd(o_gpu, lse_gpu, O_ref, LSE_ref, heads, rows):
    B, H, N, d = o_gpu.shape
    of = o_gpu.reshape(B * H, N, d)
    lf = lse_gpu.reshape(B * H, N)
    hs = list(heads)
    r = slice(None) if rows is None else list(rows)
    og = to_f64(of[hs][:, r])
    lg = to_f64(lf[hs][:, r])
    err = np.abs(og - O_ref)
    lerr = np.abs(lg - LSE_ref)
    return {
        "o_max": float(err.max()),
        "o_mean": float(err.mean()),
        "lse_max": float(lerr.max()),
        "finite": bool(np.isfinite(og).all() and np.isfinite(lg).all()),
    }


def assert_within(stats, o_max=O_MAX, o_mean=O_MEAN, lse_max=LSE_MAX):
    assert stats["finite"], stats
    assert stats["o_max"] <= o_max, stats
    assert stats["o_mean"] <= o_mean, stats
    if "lse_max" in stats:
        assert stats["lse_max"] <= lse_max, stats
