"""GPU parity of the attention backward (attn_bwd, attn_bwd_gqa) against the
fp64 oracle's chain rule ("Why Fast GPUs Still Wait for Memory",
"FlashAttention is an IO algorithm": the backward recomputes S from Q, K).

Tolerance.  The kernels round P and dS to bf16 (relative error <= 2^-9) before
the tensor-core products and accumulate in fp32, then round the gradients to
bf16 once.  Each gradient element is a sum over up to N products whose
rounding errors are independent, so the error is a few bf16 ulps of the
largest terms: relative to the tensor's largest reference magnitude, the
worst element must be within 1.5e-2 and the mean within 1.5e-3 (the O bounds
of the forward, taken relative because gradient magnitudes scale with N, d
and the mask).  Where the reference is exactly zero (one visible key: P = 1
and dS = 0) the scale floors at 1e-3: the kernel's dS = P (dP - delta), with
delta taken from the bf16 output, leaves residues far below that.
"""
import numpy as np
import pytest
import torch

import exact_attention_tma_gb300 as ea
import oracle
from exact_attention_tma_gb300.inputs import WORKLOADS, bwd_inputs, workload_inputs
from parity import to_f64

pytestmark = pytest.mark.gpu

REL_MAX = 1.5e-2
REL_MEAN = 1.5e-3


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from exact_attention_tma_gb300 import build

    build.build()
    ea.load()
    yield
    assert ea.attn_get_device_status() == 0


def _oracle_fwd(q, k, v, scale, causal):
    """O (rounded to bf16, as a forward would hand it over) and LSE (fp32)."""
    O, L = oracle.attention_gqa(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    return (torch.from_numpy(O).to(torch.bfloat16).to(q.device),
            torch.from_numpy(L).to(torch.float32).to(q.device))


def _bwd(q, k, v, o, do, lse, causal, scale):
    dq = torch.empty_like(q)
    dk = torch.empty_like(k)
    dv = torch.empty_like(v)
    ea.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, causal, scale)
    torch.cuda.synchronize()
    return dq, dk, dv


def _assert_grad_close(got, ref, name):
    ref = np.asarray(ref)
    err = np.abs(to_f64(got) - ref)
    assert np.isfinite(err).all(), name
    mag = max(np.abs(ref).max(), 1e-3)
    assert err.max() <= REL_MAX * mag, (name, err.max(), mag)
    assert err.mean() <= REL_MEAN * mag, (name, err.mean(), mag)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(2, 2), (4, 2), (3, 1)])
@pytest.mark.parametrize("N", [1, 128, 300, 520])
def test_bwd_small_full(N, H, H_kv, d, causal):
    q, k, v, do = bwd_inputs(2, H, N, d, seed=N + 3 * H + H_kv + d + causal, device="cuda",
                             H_kv=H_kv)
    scale = d ** -0.5
    o, lse = _oracle_fwd(q, k, v, scale, causal)
    dq, dk, dv = _bwd(q, k, v, o, do, lse, causal, scale)
    rq, rk, rv = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale,
                                           causal)
    _assert_grad_close(dq, rq, "dQ")
    _assert_grad_close(dk, rk, "dK")
    _assert_grad_close(dv, rv, "dV")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_after_own_forward(causal):
    # End to end: O and LSE from attn_fwd feed the backward.
    q, k, v, do = bwd_inputs(1, 2, 700, 128, seed=21, device="cuda")
    scale = 128 ** -0.5
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    ea.attn_fwd(q, k, v, o, lse, causal, scale)
    dq, dk, dv = _bwd(q, k, v, o, do, lse, causal, scale)
    rq, rk, rv = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale,
                                           causal)
    _assert_grad_close(dq, rq, "dQ")
    _assert_grad_close(dk, rk, "dK")
    _assert_grad_close(dv, rv, "dV")


def test_bwd_caller_workspace_and_run_to_run_identical():
    q, k, v, do = bwd_inputs(2, 4, 640, 64, seed=22, device="cuda", H_kv=2)
    scale = 0.125
    o, lse = _oracle_fwd(q, k, v, scale, True)
    first = _bwd(q, k, v, o, do, lse, True, scale)
    ws = torch.empty(ea.attn_bwd_workspace_bytes(2, 4, 640, 64), dtype=torch.uint8,
                     device="cuda")
    for _ in range(5):
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ea.attn_bwd_ws(q, k, v, o, do, lse, dq, dk, dv, True, scale, ws)
        torch.cuda.synchronize()
        assert torch.equal(dq, first[0]) and torch.equal(dk, first[1])
        assert torch.equal(dv, first[2])


def test_bwd_workload_sampled():
    # The full causal backward workload; the oracle recomputes a few heads
    # (first, a middle one, last) from the same inputs.
    w = WORKLOADS["causal_bwd"]
    q, k, v, do = workload_inputs(w, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    ea.attn_fwd(q, k, v, o, lse, w.causal, w.scale)
    dq, dk, dv = _bwd(q, k, v, o, do, lse, w.causal, w.scale)
    heads = [0, 37, w.B * w.H - 1]
    rq, rk, rv = oracle.attention_backward(to_f64(q), to_f64(k), to_f64(v), to_f64(do), w.scale,
                                           w.causal, heads=heads)
    for t, flat in enumerate(heads):
        b, h = divmod(flat, w.H)
        _assert_grad_close(dq[b, h], rq[t], f"dQ head {flat}")
        _assert_grad_close(dk[b, h], rk[t], f"dK head {flat}")
        _assert_grad_close(dv[b, h], rv[t], f"dV head {flat}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N,d", [(200, 128), (200, 64), (100, 128)])
def test_bwd_many_short_items_per_persistent_cta(causal, N, d):
    """Both persistent gradient kernels over far more items than SMs: (K/V
    head, key tile) items for dK/dV, with dK/dV leaving through the K/V slots
    that the next item reloads, and (query head, query tile) items for dQ,
    whose Q and dO travel through the K/V ring and enter TMEM during the
    previous item's epilogue (N = 100: one key tile per item, so Q / dO and
    K / V entries alternate in the ring; N = 200: a ragged second tile).
    Batches at the start, middle and end of the item order are checked
    against the oracle in full."""
    B, H, H_kv = 96, 4, 2   # N = 200: 192 K/V heads x 2 key tiles = 384 dK/dV items, 768 dQ items
    q, k, v, do = bwd_inputs(B, H, N, d, seed=77 + causal + N + d, device="cuda", H_kv=H_kv)
    scale = d ** -0.5
    o, lse = _oracle_fwd(q, k, v, scale, causal)
    dq, dk, dv = _bwd(q, k, v, o, do, lse, causal, scale)
    for b in (0, 47, B - 1):
        rq, rk, rv = oracle.attention_backward(to_f64(q[b:b + 1]), to_f64(k[b:b + 1]),
                                               to_f64(v[b:b + 1]), to_f64(do[b:b + 1]), scale,
                                               causal)
        _assert_grad_close(dq[b:b + 1], rq, "dQ")
        _assert_grad_close(dk[b:b + 1], rk, "dK")
        _assert_grad_close(dv[b:b + 1], rv, "dV")
