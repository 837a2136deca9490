"""GPU parity of the split-KV decode (split kernel + log-sum-exp combine)
against the fp64 oracle's unsplit decode (the definition), element by element.
"""
import numpy as np
import pytest
import torch

import exact_attention_tma_gb300 as ea
import oracle
from exact_attention_tma_gb300.inputs import WORKLOADS, decode_inputs, workload_inputs
from parity import O_MAX, O_MEAN, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from exact_attention_tma_gb300 import build

    build.build()
    ea.load()
    yield
    assert ea.attn_get_device_status() == 0


def _ref(q, K, V, scale, heads=None):
    B, H, L, d = K.shape
    hs = list(range(B * H)) if heads is None else list(heads)
    O, _ = oracle.decode(to_f64(q.reshape(B * H, d)[hs]), to_f64(K.reshape(B * H, L, d)[hs]),
                         to_f64(V.reshape(B * H, L, d)[hs]), scale)
    return O, hs


def _check(o, O_ref, hs):
    B, H, d = o.shape
    err = np.abs(to_f64(o.reshape(B * H, d)[hs]) - O_ref)
    assert np.isfinite(err).all()
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("L", [1, 2, 31, 32, 33, 100, 255, 256, 257, 1000, 4099])
def test_small_caches_full(L, d):
    B, H = 2, 3
    q, K, V = decode_inputs(B, H, L, d, seed=L + d, device="cuda")
    o = ea.decode(q, K, V, scale=d ** -0.5)
    torch.cuda.synchronize()
    O_ref, hs = _ref(q, K, V, d ** -0.5)
    _check(o, O_ref, hs)


def test_decode_workload_all_heads():
    w = WORKLOADS["decode"]
    q, K, V = workload_inputs(w, device="cuda")
    o = ea.decode(q, K, V, scale=w.scale)
    torch.cuda.synchronize()
    O_ref, hs = _ref(q, K, V, w.scale)
    _check(o, O_ref, hs)


def test_caller_workspace_matches_library_workspace():
    B, H, L, d = 3, 5, 777, 128
    q, K, V = decode_inputs(B, H, L, d, seed=5, device="cuda")
    o1 = ea.decode(q, K, V, scale=0.09)
    nbytes = ea.attn_decode_workspace_bytes(B, H, L, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    o2 = torch.empty_like(q)
    ea.attn_decode_ws(q, K, V, o2, 0.09, ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)
    with pytest.raises(ea.AttnError):
        ea.attn_decode_ws(q, K, V, o2, 0.09, ws[: nbytes - 16])


def test_peaky_scores():
    B, H, L, d = 2, 2, 3000, 64
    q, K, V = decode_inputs(B, H, L, d, seed=8, device="cuda")
    q = (q.float() * 6).to(torch.bfloat16)
    o = ea.decode(q, K, V, scale=0.125)
    torch.cuda.synchronize()
    O_ref, hs = _ref(q, K, V, 0.125)
    _check(o, O_ref, hs)


def test_concurrent_calls_on_several_streams():
    """Calls running at the same time on different streams, each with a
    workspace of its own (160 calls in flight in groups of four), each give
    exactly the result of the same call made alone."""
    B, H, L, d = 2, 16, 3000, 128
    ins = [decode_inputs(B, H, L, d, seed=50 + n, device="cuda") for n in range(4)]
    refs = [ea.decode(q, K, V, scale=d ** -0.5) for q, K, V in ins]
    torch.cuda.synchronize()
    nbytes = ea.attn_decode_workspace_bytes(B, H, L, d)
    wss = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(4)]
    outs = [torch.empty_like(q) for q, _, _ in ins]
    streams = [torch.cuda.Stream() for _ in range(4)]
    for rep in range(40):   # 160 calls in flight in groups of four
        for s, (q, K, V), o, ws in zip(streams, ins, outs, wss):
            with torch.cuda.stream(s):
                ea.attn_decode_ws(q, K, V, o, d ** -0.5, ws, stream=s)
    torch.cuda.synchronize()
    for o, ref in zip(outs, refs):
        assert torch.equal(o, ref)
    assert ea.attn_get_device_status() == 0
