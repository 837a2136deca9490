"""GPU parity of the FP8 (E4M3) forward (attn_fwd_fp8) against the fp64 oracle
of the descaled inputs ("Why Fast GPUs Still Wait for Memory": FP8 doubles the
tensor ceiling; the operation is the same attention).

Bound.  The inputs are exact E4M3 values, so the kernel's only approximation
beyond fp32 arithmetic is P: it is rounded to E4M3 as p * 2^2 with p <= 64.
A normal E4M3 value carries a relative rounding error of at most 2^-4; below
2^-6 (p < 2^-8) the absolute error is at most half the subnormal spacing,
2^-10 / 2^2 = 2^-12 in units of p.  The row sum l uses the unrounded p, so
    |O - O_ref| <= 2^-4 sum_j P_ij |V_jc| + 2^-12 sum_j |V_jc| / l_i
                   + 2^-8 |O_ref| (bf16 output rounding) + 1e-5,
with P the exact normalised softmax and l_i = 1 / max_j P_ij the exact row sum
(the kernel's l is at least that).  Checked element by element; the LSE
(fp32, computed from the unrounded p) within 1e-3.
"""
import numpy as np
import pytest
import torch

import exact_attention_tma_gb300 as ea
import oracle
from exact_attention_tma_gb300.inputs import WORKLOADS, fp8_inputs, workload_inputs
from parity import LSE_MAX, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from exact_attention_tma_gb300 import build

    build.build()
    ea.load()
    yield
    assert ea.attn_get_device_status() == 0


def _codes(t):
    return t.view(torch.uint8).cpu().numpy()


def _run(q8, k8, v8, ds, causal, scale):
    B, H, N, d = q8.shape
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    ea.attn_fwd_fp8(q8, k8, v8, o, lse, causal, scale, *ds)
    torch.cuda.synchronize()
    return o, lse


def _check_head(o, lse, Q, K, V, scale, causal, rows=None):
    """o, lse: kernel output rows of one head; Q, K, V: fp64 descaled inputs."""
    O_ref, L_ref, P, _ = oracle.attention_head(Q, K, V, scale, causal, rows=rows, return_p=True)
    absV = np.abs(V)
    l_row = 1.0 / P.max(axis=1)
    bound = (2.0 ** -4) * (P @ absV) + (2.0 ** -12) * absV.sum(0)[None, :] / l_row[:, None] \
        + (2.0 ** -8) * np.abs(O_ref) + 1e-5
    err = np.abs(to_f64(o) - O_ref)
    assert np.isfinite(err).all()
    worst = (err / bound).max()
    assert worst <= 1.0, worst
    lerr = np.abs(to_f64(lse) - L_ref).max()
    assert lerr <= LSE_MAX, lerr
    return worst


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 64, 128, 300, 520])
def test_fp8_small_full(N, causal):
    (q8, k8, v8), ds = fp8_inputs(2, 2, N, 128, seed=N + causal, device="cuda")
    scale = 128 ** -0.5
    o, lse = _run(q8, k8, v8, ds, causal, scale)
    qc, kc, vc = _codes(q8), _codes(k8), _codes(v8)
    for b in range(2):
        for h in range(2):
            _check_head(o[b, h], lse[b, h], oracle.decode_e4m3(qc[b, h]) * ds[0],
                        oracle.decode_e4m3(kc[b, h]) * ds[1], oracle.decode_e4m3(vc[b, h]) * ds[2],
                        scale, causal)


def test_fp8_workload_sampled():
    w = WORKLOADS["fp8_causal_fwd"]
    (q8, k8, v8), ds = workload_inputs(w, device="cuda")
    o, lse = _run(q8, k8, v8, ds, w.causal, w.scale)
    rows = [0, 1, 127, 128, 129, 1000, 2047]
    for flat in [0, 37, w.B * w.H - 1]:
        b, h = divmod(flat, w.H)
        Q = oracle.decode_e4m3(_codes(q8[b, h])) * ds[0]
        K = oracle.decode_e4m3(_codes(k8[b, h])) * ds[1]
        V = oracle.decode_e4m3(_codes(v8[b, h])) * ds[2]
        _check_head(o[b, h, rows], lse[b, h, rows], Q, K, V, w.scale, w.causal, rows=rows)
