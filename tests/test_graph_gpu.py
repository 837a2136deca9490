"""CUDA-graph capture of the C-ABI calls (GPU).

Decode steps are short, so serving code captures them in CUDA graphs to
remove launch overhead.  Every entry point here launches on the caller's
stream with no host synchronisation and no allocation once warmed up (the
library workspace grows only on first use, and caller-owned workspaces
never allocate), so a captured graph replays the same kernels.  Each test
warms up outside the capture, captures one call, writes new inputs into the
captured buffers and checks the replay against a direct call.
"""
import pytest
import torch

import exact_attention_tma_gb300 as ea
from exact_attention_tma_gb300.inputs import bwd_inputs, decode_inputs, paged_decode_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from exact_attention_tma_gb300 import build

    build.build()
    ea.load()
    yield
    assert ea.attn_get_device_status() == 0


def _capture(fn):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn(s)                      # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn(s)
    return g


def test_graph_replays_decode_and_grouped_decode():
    q, K, V = decode_inputs(4, 16, 3000, 128, seed=41, device="cuda", H_kv=4)
    ws = torch.empty(ea.attn_decode_workspace_bytes(4, 16, 3000, 128), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty_like(q)
    g = _capture(lambda s: ea.attn_decode_gqa_ws(q, K, V, o, 0.1, ws, stream=s))
    q2, K2, V2 = decode_inputs(4, 16, 3000, 128, seed=42, device="cuda", H_kv=4)
    q.copy_(q2), K.copy_(K2), V.copy_(V2)
    g.replay()
    torch.cuda.synchronize()
    ref = torch.empty_like(q)
    ea.attn_decode_gqa_ws(q2, K2, V2, ref, 0.1, ws)
    torch.cuda.synchronize()
    assert torch.equal(o, ref)


def test_graph_replays_paged_decode_and_forward():
    q, Kp, Vp, table, sl = paged_decode_inputs(2, 8, 500, 128, 64, seed=43, device="cuda",
                                               H_kv=2)
    o = torch.empty_like(q)
    qf, kf, vf, _ = bwd_inputs(2, 4, 384, 64, seed=44, device="cuda")
    of = torch.empty_like(qf)
    lse = torch.empty(qf.shape[:3], dtype=torch.float32, device="cuda")

    def step(s):
        ea.attn_decode_paged(q, Kp, Vp, table, sl, o, 0.1, stream=s)
        ea.attn_fwd(qf, kf, vf, of, lse, True, 0.125, stream=s)

    g = _capture(step)
    perm = torch.randperm(table.numel(), generator=torch.Generator().manual_seed(3))
    table.copy_(table.flatten()[perm.to(table.device)].view_as(table))
    qf.mul_(0.5)
    g.replay()
    torch.cuda.synchronize()
    o_ref, of_ref = torch.empty_like(o), torch.empty_like(of)
    l_ref = torch.empty_like(lse)
    ea.attn_decode_paged(q, Kp, Vp, table, sl, o_ref, 0.1)
    ea.attn_fwd(qf, kf, vf, of_ref, l_ref, True, 0.125)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(of, of_ref) and torch.equal(lse, l_ref)


def test_graph_replays_backward():
    q, k, v, do = bwd_inputs(1, 4, 300, 128, seed=45, device="cuda", H_kv=2)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    ea.attn_fwd_gqa(q, k, v, o, lse, True, 0.09)
    ws = torch.empty(ea.attn_bwd_workspace_bytes(1, 4, 300, 128), dtype=torch.uint8,
                     device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    g = _capture(lambda s: ea.attn_bwd_ws(q, k, v, o, do, lse, dq, dk, dv, True, 0.09, ws,
                                          stream=s))
    do.mul_(-2.0)
    g.replay()
    torch.cuda.synchronize()
    r = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    ea.attn_bwd_ws(q, k, v, o, do, lse, *r, True, 0.09, ws)
    torch.cuda.synchronize()
    assert torch.equal(dq, r[0]) and torch.equal(dk, r[1]) and torch.equal(dv, r[2])


def test_graph_replays_fp8_forward():
    """The FP8 forward is two launches, the second a dependent launch that
    may start before the V transpose has finished; captured, it replays to
    the result of a direct call."""
    from exact_attention_tma_gb300.inputs import fp8_inputs

    (q8, k8, v8), ds = fp8_inputs(2, 4, 700, 128, seed=46, device="cuda")
    o = torch.empty(q8.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(q8.shape[:3], dtype=torch.float32, device="cuda")
    g = _capture(lambda s: ea.attn_fwd_fp8(q8, k8, v8, o, lse, True, 0.09, *ds, stream=s))
    (q2, k2, v2), _ = fp8_inputs(2, 4, 700, 128, seed=47, device="cuda")
    q8.copy_(q2), k8.copy_(k2), v8.copy_(v2)
    g.replay()
    torch.cuda.synchronize()
    o_ref, l_ref = torch.empty_like(o), torch.empty_like(lse)
    ea.attn_fwd_fp8(q8, k8, v8, o_ref, l_ref, True, 0.09, *ds)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
