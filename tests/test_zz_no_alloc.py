"""attn_decode_noalloc: decode for callers that cannot allocate device memory.

Some hosts cannot let a library call cudaMalloc: their own allocator already
holds the GPU's memory, an allocation could block or synchronise the device at
a bad moment, or the host forbids plug-ins from allocating.  For them the
library keeps a fixed scratch array in device memory and attn_decode_noalloc
uses it instead of allocating a workspace.  These tests call that entry point
through the C ABI and check that two calls in a row give the same output as
the allocating attn_decode, within the tolerance of the other decode tests, and
that a shape too large for the scratch is refused before anything runs.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_tma_gb300 as ea
from exact_attention_tma_gb300.inputs import decode_inputs
import oracle
from parity import O_MAX, O_MEAN, to_f64

pytestmark = pytest.mark.gpu

NOMEM = 6


@pytest.fixture(scope="module")
def lib(cuda_ok):
    from exact_attention_tma_gb300 import build

    build.build()
    return ea.load()


def _call_noalloc(lib, q, K, V, O, scale):
    B, H, L, d = K.shape
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    return lib.attn_decode_noalloc(vp(q.data_ptr()), vp(K.data_ptr()), vp(V.data_ptr()),
                                   vp(O.data_ptr()), B, H, L, d, float(scale), stream)


def _close(a, b):
    err = (a.double() - b.double()).abs()
    assert torch.isfinite(a.double()).all()
    assert err.max().item() <= O_MAX and err.mean().item() <= O_MEAN, (err.max(), err.mean())


def _matches_oracle(out, q, K, V, scale):
    """Element by element against the fp64 oracle (independent of both decode paths)."""
    O_ref, _ = oracle.decode(to_f64(q), to_f64(K), to_f64(V), scale)
    err = np.abs(to_f64(out) - O_ref)
    assert np.isfinite(to_f64(out)).all()
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())


@pytest.mark.parametrize("shape", [(4, 8, 1500, 128), (2, 5, 333, 64)])
def test_noalloc_matches_allocating_decode_on_two_calls(lib, shape):
    B, H, L, d = shape
    scale = d ** -0.5
    for call, seed in enumerate((40, 41)):
        q, K, V = decode_inputs(B, H, L, d, seed=seed, device="cuda")
        ref = ea.decode(q, K, V, scale=scale)
        out = torch.full_like(q, float("nan"))
        assert _call_noalloc(lib, q, K, V, out, scale) == 0, f"call {call}"
        torch.cuda.synchronize()
        _close(out, ref)
        _matches_oracle(out, q, K, V, scale)
    assert ea.attn_get_device_status() == 0


def test_noalloc_refuses_shapes_beyond_its_scratch(lib):
    # 64*32 heads * 32 splits * 129 floats * 4 B = 33.8 MB > 16 MiB: refused, nothing launched.
    B, H, L, d = 64, 32, 16, 128
    q = torch.zeros((1,), dtype=torch.bfloat16, device="cuda")
    vp = ctypes.c_void_p
    p = vp(q.data_ptr())
    assert lib.attn_decode_noalloc(p, p, p, p, B, H, L, d, 0.1, None) == NOMEM
    # Largest shape that fits still runs: 1016 heads at d = 128.
    assert ea.attn_decode_workspace_bytes(8, 127, 64, 128) <= 16 << 20
    q, K, V = decode_inputs(8, 127, 64, 128, seed=3, device="cuda")
    out = torch.empty_like(q)
    assert _call_noalloc(lib, q, K, V, out, 128 ** -0.5) == 0
    torch.cuda.synchronize()
    _close(out, ea.decode(q, K, V, scale=128 ** -0.5))
    assert np.isfinite(out.float().cpu().numpy()).all()


def test_noalloc_head_limit_at_d64(lib):
    # At d = 64 the 16 MiB scratch holds 2016 heads (2016 * 32 * 65 * 4 B); 2017 are refused.
    assert ea.attn_decode_workspace_bytes(1, 2016, 64, 64) <= 16 << 20
    assert ea.attn_decode_workspace_bytes(1, 2017, 64, 64) > 16 << 20
    q, K, V = decode_inputs(1, 2016, 64, 64, seed=5, device="cuda")
    out = torch.full_like(q, float("nan"))
    assert _call_noalloc(lib, q, K, V, out, 0.125) == 0
    torch.cuda.synchronize()
    _matches_oracle(out, q, K, V, 0.125)
    q1, K1, V1 = decode_inputs(1, 2017, 64, 64, seed=5, device="cuda")
    untouched = torch.full_like(q1, 7.0)
    assert _call_noalloc(lib, q1, K1, V1, untouched, 0.125) == NOMEM
    torch.cuda.synchronize()
    assert (untouched == 7.0).all()   # nothing was launched
    assert ea.attn_get_device_status() == 0
