"""Largest-size GPU checks: every tensor here holds more than 2^31 elements, so
any 32-bit index arithmetic in a kernel would address the wrong rows of the
last heads.  Inputs are drawn on the device (seeded bf16 normals); the fp64
oracle recomputes the first and the last head (sampled rows for the forward),
which sit at the two ends of the index space.
"""
import numpy as np
import pytest
import torch

import exact_attention_tma_gb300 as ea
import oracle
from parity import LSE_MAX, O_MAX, O_MEAN, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from exact_attention_tma_gb300 import build

    build.build()
    ea.load()
    yield
    torch.cuda.empty_cache()
    assert ea.attn_get_device_status() == 0


def _randn(shape, gen):
    return torch.randn(shape, generator=gen, device="cuda", dtype=torch.bfloat16)


def _close(o, ref):
    err = np.abs(to_f64(o) - ref)
    assert np.isfinite(err).all()
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()


def test_forward_beyond_2_31_elements():
    B, H, N, d = 72, 32, 8192, 128
    assert B * H * N * d > 2 ** 31
    g = torch.Generator(device="cuda").manual_seed(101)
    q, k, v = _randn((B, H, N, d), g), _randn((B, H, N, d), g), _randn((B, H, N, d), g)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ea.attn_fwd(q, k, v, o, lse, True, d ** -0.5)
    torch.cuda.synchronize()
    rows = [0, 1, 127, 128, 4095, 8190, 8191]
    for b, h in [(0, 0), (B - 1, H - 1)]:
        O_ref, L_ref = oracle.attention_head(to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h]),
                                             d ** -0.5, True, rows=rows)
        _close(o[b, h, rows], O_ref)
        assert np.abs(to_f64(lse[b, h, rows]) - L_ref).max() <= LSE_MAX
    del q, k, v, o, lse
    torch.cuda.empty_cache()


def test_decode_beyond_2_31_elements():
    B, H, L, d = 16, 32, 65536, 128
    assert B * H * L * d > 2 ** 31
    g = torch.Generator(device="cuda").manual_seed(102)
    q, K, V = _randn((B, H, d), g), _randn((B, H, L, d), g), _randn((B, H, L, d), g)
    o = torch.empty_like(q)
    ea.attn_decode(q, K, V, o, d ** -0.5)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (B - 1, H - 1)]:
        O_ref, _ = oracle.decode(to_f64(q[b, h]), to_f64(K[b, h]), to_f64(V[b, h]), d ** -0.5)
        _close(o[b, h], O_ref)
    del q, K, V, o
    torch.cuda.empty_cache()


def test_grouped_decode_beyond_2_31_elements():
    B, H, H_kv, L, d = 16, 64, 8, 196608, 128
    assert B * H_kv * L * d > 2 ** 31
    g = torch.Generator(device="cuda").manual_seed(103)
    q, K, V = _randn((B, H, d), g), _randn((B, H_kv, L, d), g), _randn((B, H_kv, L, d), g)
    o = torch.empty_like(q)
    ea.attn_decode_gqa(q, K, V, o, d ** -0.5)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (B - 1, H - 1)]:
        kh = oracle.kv_head_of(h, H, H_kv)
        O_ref, _ = oracle.decode(to_f64(q[b, h]), to_f64(K[b, kh]), to_f64(V[b, kh]), d ** -0.5)
        _close(o[b, h], O_ref)
    del q, K, V, o
    torch.cuda.empty_cache()


def test_backward_beyond_2_31_elements():
    B, H, N, d = 640, 32, 1024, 128
    assert B * H * N * d > 2 ** 31
    g = torch.Generator(device="cuda").manual_seed(104)
    q, k, v, do = (_randn((B, H, N, d), g) for _ in range(4))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ea.attn_fwd(q, k, v, o, lse, True, d ** -0.5)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ea.attn_bwd(q, k, v, o, do, lse, dq, dk, dv, True, d ** -0.5)
    torch.cuda.synchronize()
    for b, h in [(0, 0), (B - 1, H - 1)]:
        rq, rk, rv = oracle.attention_backward_head(to_f64(q[b, h]), to_f64(k[b, h]),
                                                    to_f64(v[b, h]), to_f64(do[b, h]),
                                                    d ** -0.5, True)
        for got, ref in ((dq[b, h], rq), (dk[b, h], rk), (dv[b, h], rv)):
            err = np.abs(to_f64(got) - ref)
            mag = np.abs(ref).max()
            assert err.max() <= 1.5e-2 * mag and err.mean() <= 1.5e-3 * mag
    del q, k, v, do, o, lse, dq, dk, dv
    torch.cuda.empty_cache()


def test_fp8_forward_beyond_2_31_elements():
    B, H, N, d = 72, 32, 8192, 128
    assert B * H * N * d > 2 ** 31
    g = torch.Generator(device="cuda").manual_seed(105)
    q8, k8, v8 = ((_randn((B, H, N, d), g).float() * 32).clamp(-448, 448).to(torch.float8_e4m3fn)
                  for _ in range(3))
    ds = (1 / 32, 1 / 32, 1 / 32)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ea.attn_fwd_fp8(q8, k8, v8, o, lse, True, d ** -0.5, *ds)
    torch.cuda.synchronize()
    rows = [0, 1, 128, 4095, 8191]
    for b, h in [(0, 0), (B - 1, H - 1)]:
        Q, K, V = (oracle.decode_e4m3(t[b, h].view(torch.uint8).cpu().numpy()) * s
                   for t, s in ((q8, ds[0]), (k8, ds[1]), (v8, ds[2])))
        O_ref, L_ref, P, _ = oracle.attention_head(Q, K, V, d ** -0.5, True, rows=rows,
                                                   return_p=True)
        # The FP8 bound of test_fp8_gpu: P rounded to E4M3.
        absV = np.abs(V)
        bound = (2.0 ** -4) * (P @ absV) + (2.0 ** -12) * absV.sum(0)[None, :] * P.max(1)[:, None] \
            + (2.0 ** -8) * np.abs(O_ref) + 1e-5
        assert (np.abs(to_f64(o[b, h, rows]) - O_ref) <= bound).all()
        assert np.abs(to_f64(lse[b, h, rows]) - L_ref).max() <= LSE_MAX
    del q8, k8, v8, o, lse
    torch.cuda.empty_cache()
