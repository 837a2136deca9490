"""GPU parity of grouped-query attention (attn_fwd_gqa, attn_decode_gqa)
against the fp64 oracle ("Why Fast GPUs Still Wait for Memory", Attention III:
h query heads over h_kv K/V heads, query head h reading K/V head floor(h / g)).
"""
import numpy as np
import pytest
import torch

import exact_attention_tma_gb300 as ea
import oracle
from exact_attention_tma_gb300.inputs import WORKLOADS, decode_inputs, fwd_inputs, workload_inputs
from parity import LSE_MAX, O_MAX, O_MEAN, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from exact_attention_tma_gb300 import build

    build.build()
    ea.load()
    yield
    assert ea.attn_get_device_status() == 0


def _fwd(q, k, v, causal, scale):
    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    ea.attn_fwd_gqa(q, k, v, o, lse, causal, scale)
    torch.cuda.synchronize()
    return o, lse


def _assert_close(o, O_ref, lse=None, LSE_ref=None):
    err = np.abs(to_f64(o) - O_ref)
    assert np.isfinite(err).all()
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    if lse is not None:
        lerr = np.abs(to_f64(lse) - LSE_ref)
        assert lerr.max() <= LSE_MAX, lerr.max()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(4, 1), (4, 2), (8, 2), (6, 3)])
@pytest.mark.parametrize("N", [128, 300])
def test_fwd_small_full(N, H, H_kv, d, causal):
    q, k, v = fwd_inputs(2, H, N, d, seed=N + H + H_kv + d, device="cuda", H_kv=H_kv)
    scale = d ** -0.5
    o, lse = _fwd(q, k, v, causal, scale)
    O_ref, LSE_ref = oracle.attention_gqa(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    _assert_close(o, O_ref, lse, LSE_ref)


def test_fwd_one_group_matches_multi_head_call():
    q, k, v = fwd_inputs(2, 4, 300, 128, seed=7, device="cuda")
    o1, l1 = _fwd(q, k, v, True, 128 ** -0.5)
    o2 = torch.empty_like(q)
    l2 = torch.empty_like(l1)
    ea.attn_fwd(q, k, v, o2, l2, True, 128 ** -0.5)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_fwd_gqa_workload_sampled():
    w = WORKLOADS["gqa_fwd"]
    q, k, v = workload_inputs(w, device="cuda")
    o, lse = _fwd(q, k, v, w.causal, w.scale)
    rows = [0, 1, 127, 128, 1000, 2047]
    for flat in [0, 7, 8, 63, 64 + 31, 3 * 64 + 56, w.B * w.H - 1]:
        b, h = divmod(flat, w.H)
        kh = oracle.kv_head_of(h, w.H, w.H_kv)
        O_ref, LSE_ref = oracle.attention_head(to_f64(q[b, h]), to_f64(k[b, kh]), to_f64(v[b, kh]),
                                               w.scale, w.causal, rows=rows)
        _assert_close(o[b, h, rows], O_ref, lse[b, h, rows], LSE_ref)


def _dec(q, K, V, scale):
    o = torch.empty_like(q)
    ea.attn_decode_gqa(q, K, V, o, scale)
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(8, 1), (8, 2), (8, 4), (12, 4), (16, 2), (32, 2)])
@pytest.mark.parametrize("L", [1, 33, 257, 1000])
def test_decode_small_full(L, H, H_kv, d):
    q, K, V = decode_inputs(2, H, L, d, seed=L + H + H_kv + d, device="cuda", H_kv=H_kv)
    o = _dec(q, K, V, d ** -0.5)
    O_ref, _ = oracle.decode_gqa(to_f64(q), to_f64(K), to_f64(V), d ** -0.5)
    _assert_close(o, O_ref)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(16, 1), (20, 1), (24, 1), (64, 2)])
@pytest.mark.parametrize("L", [5, 5000])
def test_decode_large_groups_and_multi_tile_splits(L, H, H_kv, d):
    # Groups of more than 16 query heads span several CTAs (16 rows each, the
    # last one ragged); L = 5000 gives splits of several 64-key tiles with a
    # ragged last tile.
    q, K, V = decode_inputs(1, H, L, d, seed=L + H + d, device="cuda", H_kv=H_kv)
    o = _dec(q, K, V, d ** -0.5)
    O_ref, _ = oracle.decode_gqa(to_f64(q), to_f64(K), to_f64(V), d ** -0.5)
    _assert_close(o, O_ref)


@pytest.mark.parametrize("H,H_kv", [(128, 8), (64, 8)])
def test_decode_gqa_run_to_run_identical(H, H_kv):
    # Every launch must give the same bits: the K/V stages are rewritten by
    # TMA while other warps may still be reading the previous tile, so any
    # ordering gap between the readers and the refill shows up here first.
    q, K, V = decode_inputs(16, H, 8192, 128, seed=11, device="cuda", H_kv=H_kv)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    first = None
    for _ in range(40):
        flush.zero_()
        ea.attn_decode_gqa(q, K, V, o, 128 ** -0.5)
        if first is None:
            first = o.clone()
        else:
            assert torch.equal(o, first)
    torch.cuda.synchronize()


@pytest.mark.parametrize("B,H,H_kv,L,d", [(1, 16, 1, 5000, 64), (2, 8, 2, 70000, 128),
                                          (3, 24, 1, 999, 128), (1, 64, 8, 300, 64)])
def test_decode_gqa_writes_only_its_workspace(B, H, H_kv, L, d):
    # The caller's workspace is exactly attn_decode_workspace_bytes long and
    # followed by a guard region that must come back untouched.
    q, K, V = decode_inputs(B, H, L, d, seed=L + H, device="cuda", H_kv=H_kv)
    need = ea.attn_decode_workspace_bytes(B, H, L, d)
    guard = 1 << 16
    buf = torch.full((need + guard,), 0x5A, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    ea.attn_decode_gqa_ws(q, K, V, o, d ** -0.5, buf[:need])
    torch.cuda.synchronize()
    assert bool((buf[need:] == 0x5A).all())
    O_ref, _ = oracle.decode_gqa(to_f64(q), to_f64(K), to_f64(V), d ** -0.5)
    _assert_close(o, O_ref)


def test_decode_gqa_with_caller_workspace_matches():
    q, K, V = decode_inputs(2, 16, 700, 128, seed=3, device="cuda", H_kv=4)
    o1 = _dec(q, K, V, 0.1)
    ws = torch.empty(ea.attn_decode_workspace_bytes(2, 16, 700, 128), dtype=torch.uint8,
                     device="cuda")
    o2 = torch.empty_like(q)
    ea.attn_decode_gqa_ws(q, K, V, o2, 0.1, ws)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


def test_decode_gqa_workload_sampled():
    w = WORKLOADS["gqa_decode"]
    q, K, V = workload_inputs(w, device="cuda")
    o = _dec(q, K, V, w.scale)
    for flat in [0, 1, 7, 8, 63, 5 * 64 + 9, w.B * w.H - 1]:
        b, h = divmod(flat, w.H)
        kh = oracle.kv_head_of(h, w.H, w.H_kv)
        O_ref, _ = oracle.decode(to_f64(q[b, h]), to_f64(K[b, kh]), to_f64(V[b, kh]), w.scale)
        _assert_close(o[b, h], O_ref)
