"""Host-side tests of the C ABI (no GPU needed).

The library must load and export every function include/exact_attn.h
declares, and every invalid call must be rejected by host validation with the
documented status code before any CUDA call or launch happens (so fake,
never-dereferenced pointers are enough here).
"""
import ctypes
import os
import re

import pytest

import exact_attention_tma_gb300 as ea
from exact_attention_tma_gb300 import build as ea_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

OK, NULL, SHAPE, HEADDIM, ALIGN, CUDA, NOMEM, TIMEOUT, ARG = range(9)
P = 0x10000  # fake 16-byte-aligned device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    ea_build.build()
    return ea.load()


def _declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(attn_\w+)\s*\(", text, re.M):
            names.add(m.group(1))
    return names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"attn_fwd", "attn_decode", "attn_decode_ws", "attn_get_device_status",
            "attn_status_string", "attn_decode_workspace_bytes",
            "attn_decode_num_splits", "attn_fwd_gqa", "attn_decode_gqa",
            "attn_decode_gqa_ws", "attn_decode_paged", "attn_bwd", "attn_bwd_gqa",
            "attn_bwd_gqa_ws", "attn_bwd_workspace_bytes", "attn_fwd_fp8", "attn_fwd_fp8_ws",
            "attn_fwd_fp8_workspace_bytes"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    for code in range(9):
        s = ea.attn_status_string(code)
        assert isinstance(s, str) and s
    assert ea.attn_status_string(99) == "unknown status"


def test_decode_workspace_bytes(lib):
    nsplit = ea.attn_decode_num_splits()
    assert nsplit == 32
    assert ea.attn_decode_workspace_bytes(16, 32, 8192, 128) == 16 * 32 * nsplit * (128 + 1) * 4
    assert ea.attn_decode_workspace_bytes(1, 1, 1, 64) == nsplit * 65 * 4
    assert ea.attn_decode_workspace_bytes(1, 1, 1, 96) == 0
    assert ea.attn_decode_workspace_bytes(0, 1, 1, 64) == 0


def _fwd(lib, Q=P, K=P, V=P, O=P, L=P, B=1, H=1, N=128, d=64, scale=0.125, causal=0):
    vp = ctypes.c_void_p
    return lib.attn_fwd(vp(Q), vp(K), vp(V), vp(O), vp(L), B, H, N, d, scale, causal, None)


def _dec(lib, q=P, K=P, V=P, O=P, B=1, H=1, L=128, d=64, scale=0.125):
    vp = ctypes.c_void_p
    return lib.attn_decode(vp(q), vp(K), vp(V), vp(O), B, H, L, d, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Q=0), NULL), (dict(K=0), NULL), (dict(V=0), NULL), (dict(O=0), NULL),
    (dict(L=0), NULL),
    (dict(B=0), SHAPE), (dict(H=-1), SHAPE), (dict(N=0), SHAPE), (dict(N=(1 << 24) + 1), SHAPE),
    (dict(B=1 << 13, H=1 << 12), SHAPE),
    (dict(d=96), HEADDIM), (dict(d=256), HEADDIM), (dict(d=0), HEADDIM),
    (dict(Q=P + 8), ALIGN), (dict(K=P + 2), ALIGN), (dict(V=P + 4), ALIGN),
    (dict(O=P + 1), ALIGN), (dict(L=P + 2), ALIGN),
    (dict(scale=0.0), ARG), (dict(scale=-1.0), ARG), (dict(scale=float("nan")), ARG),
    (dict(scale=float("inf")), ARG), (dict(causal=2), ARG),
])
def test_fwd_rejects_bad_arguments_before_launch(lib, kw, code):
    assert _fwd(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), NULL), (dict(K=0), NULL), (dict(V=0), NULL), (dict(O=0), NULL),
    (dict(B=0), SHAPE), (dict(L=0), SHAPE), (dict(L=(1 << 24) + 1), SHAPE),
    (dict(d=32), HEADDIM),
    (dict(q=P + 8), ALIGN), (dict(K=P + 8), ALIGN), (dict(V=P + 8), ALIGN), (dict(O=P + 2), ALIGN),
    (dict(scale=0.0), ARG), (dict(scale=float("nan")), ARG),
])
def test_decode_rejects_bad_arguments_before_launch(lib, kw, code):
    assert _dec(lib, **kw) == code
    # The allocation-free decode runs the same checks first (before its size
    # limit and its symbol lookup, so no CUDA call is made on this GPU-less host).
    assert _dec_noalloc(lib, **kw) == code


def _dec_noalloc(lib, q=P, K=P, V=P, O=P, B=1, H=1, L=128, d=64, scale=0.125):
    vp = ctypes.c_void_p
    return lib.attn_decode_noalloc(vp(q), vp(K), vp(V), vp(O), B, H, L, d, scale, None)


@pytest.mark.parametrize("kw,code", [
    # Too large for the 16 MiB scratch, with another error that must win.
    (dict(B=64, H=32, d=128, q=0), NULL), (dict(B=64, H=32, d=128, scale=float("nan")), ARG),
    (dict(B=64, H=32, d=128, O=P + 2), ALIGN), (dict(B=64, H=32, d=96), HEADDIM),
    # Valid but too large: refused before any CUDA call.
    (dict(B=64, H=32, d=128), NOMEM), (dict(B=1, H=1017, d=128), NOMEM),
    (dict(B=1, H=2017, d=64), NOMEM), (dict(B=7, H=289, d=64), NOMEM),
])
def test_decode_noalloc_checks_arguments_before_its_size_limit(lib, kw, code):
    assert _dec_noalloc(lib, **kw) == code


def test_decode_ws_checks_workspace(lib):
    vp = ctypes.c_void_p
    need = ea.attn_decode_workspace_bytes(2, 3, 100, 128)
    assert lib.attn_decode_ws(vp(P), vp(P), vp(P), vp(P), 2, 3, 100, 128, 0.1, None, need,
                              None) == NULL
    assert lib.attn_decode_ws(vp(P), vp(P), vp(P), vp(P), 2, 3, 100, 128, 0.1, vp(P + 4), need,
                              None) == ALIGN
    assert lib.attn_decode_ws(vp(P), vp(P), vp(P), vp(P), 2, 3, 100, 128, 0.1, vp(P), need - 1,
                              None) == NOMEM


@pytest.mark.parametrize("limit_ms", [0, -5, 10001])
def test_selftest_rejects_bad_limit_before_launch(lib, limit_ms):
    assert lib.attn_selftest_bounded_wait(limit_ms, None) == ARG


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(ea, "_lib", None)
    monkeypatch.setattr(ea, "_LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        ea.load()


@pytest.mark.parametrize("H,H_kv,code", [(8, 0, SHAPE), (8, 3, SHAPE), (8, -2, SHAPE), (6, 4, SHAPE)])
def test_gqa_rejects_bad_group_before_launch(lib, H, H_kv, code):
    vp = ctypes.c_void_p
    assert lib.attn_fwd_gqa(vp(P), vp(P), vp(P), vp(P), vp(P), 1, H, H_kv, 128, 64, 0.125, 0,
                            None) == code
    assert lib.attn_decode_gqa(vp(P), vp(P), vp(P), vp(P), 1, H, H_kv, 128, 64, 0.125,
                               None) == code
    assert lib.attn_decode_gqa_ws(vp(P), vp(P), vp(P), vp(P), 1, H, H_kv, 128, 64, 0.125, vp(P),
                                  1 << 20, None) == code


def test_gqa_validates_like_the_multi_head_calls(lib):
    vp = ctypes.c_void_p
    assert lib.attn_fwd_gqa(vp(0), vp(P), vp(P), vp(P), vp(P), 1, 8, 2, 128, 64, 0.125, 0,
                            None) == NULL
    assert lib.attn_fwd_gqa(vp(P), vp(P + 8), vp(P), vp(P), vp(P), 1, 8, 2, 128, 64, 0.125, 0,
                            None) == ALIGN
    assert lib.attn_fwd_gqa(vp(P), vp(P), vp(P), vp(P), vp(P), 1, 8, 2, 128, 96, 0.125, 0,
                            None) == HEADDIM
    assert lib.attn_decode_gqa(vp(P), vp(P), vp(P), vp(P), 1, 8, 2, 0, 64, 0.125, None) == SHAPE
    need = ea.attn_decode_workspace_bytes(1, 8, 100, 64)
    assert lib.attn_decode_gqa_ws(vp(P), vp(P), vp(P), vp(P), 1, 8, 2, 100, 64, 0.125, vp(P),
                                  need - 1, None) == NOMEM


def _paged(lib, q=P, Kp=P, Vp=P, bt=P, sl=P, O=P, B=2, H=4, H_kv=2, num_pages=8, page_size=16,
           max_blocks=4, d=64, scale=0.125):
    vp = ctypes.c_void_p
    return lib.attn_decode_paged(vp(q), vp(Kp), vp(Vp), vp(bt), vp(sl), vp(O), B, H, H_kv,
                                 num_pages, page_size, max_blocks, d, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), NULL), (dict(bt=0), NULL), (dict(sl=0), NULL), (dict(Vp=0), NULL),
    (dict(page_size=12), SHAPE), (dict(page_size=0), SHAPE), (dict(page_size=1 << 17), SHAPE),
    (dict(num_pages=0), SHAPE), (dict(max_blocks=0), SHAPE), (dict(H_kv=3), SHAPE),
    (dict(max_blocks=1 << 20, page_size=1 << 5), SHAPE),
    (dict(d=96), HEADDIM), (dict(Kp=P + 8), ALIGN), (dict(bt=P + 2), ALIGN),
    (dict(sl=P + 1), ALIGN), (dict(scale=float("nan")), ARG),
])
def test_paged_decode_rejects_bad_arguments_before_launch(lib, kw, code):
    assert _paged(lib, **kw) == code


def _fp8(lib, Q=P, K=P, V=P, O=P, L=P, B=1, H=2, N=300, d=128, scale=0.1, dq=0.01, dk=0.02,
         dv=0.03, causal=1):
    vp = ctypes.c_void_p
    return lib.attn_fwd_fp8(vp(Q), vp(K), vp(V), vp(O), vp(L), B, H, N, d, scale, dq, dk, dv,
                            causal, None)


@pytest.mark.parametrize("kw,code", [
    (dict(Q=0), NULL), (dict(V=0), NULL), (dict(L=0), NULL),
    (dict(N=0), SHAPE), (dict(B=0), SHAPE),
    (dict(d=64), HEADDIM), (dict(d=96), HEADDIM),
    (dict(Q=P + 8), ALIGN), (dict(O=P + 2), ALIGN), (dict(L=P + 2), ALIGN),
    (dict(scale=0.0), ARG), (dict(dq=0.0), ARG), (dict(dk=-1.0), ARG),
    (dict(dv=float("inf")), ARG), (dict(causal=3), ARG),
])
def test_fp8_fwd_rejects_bad_arguments_before_launch(lib, kw, code):
    assert _fp8(lib, **kw) == code


def test_fp8_workspace_bytes(lib):
    # V^T: d x N_pad bytes per head, N_pad = N rounded up to 16.
    assert ea.attn_fwd_fp8_workspace_bytes(2, 3, 300, 128) == 2 * 3 * 128 * 304
    assert ea.attn_fwd_fp8_workspace_bytes(2, 3, 300, 64) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(Q=0), NULL), (dict(dO=0), NULL), (dict(dV=0), NULL), (dict(LSE=0), NULL),
    (dict(H_kv=3), SHAPE), (dict(N=0), SHAPE), (dict(d=96), HEADDIM),
    (dict(dO=P + 8), ALIGN), (dict(dK=P + 4), ALIGN), (dict(LSE=P + 2), ALIGN),
    (dict(scale=float("nan")), ARG), (dict(causal=2), ARG),
])
def test_bwd_rejects_bad_arguments_before_launch(lib, kw, code):
    vp = ctypes.c_void_p
    a = dict(Q=P, K=P, V=P, O=P, dO=P, LSE=P, dQ=P, dK=P, dV=P, B=1, H=4, H_kv=2, N=300, d=64,
             scale=0.125, causal=1)
    a.update(kw)
    assert lib.attn_bwd_gqa(*(vp(a[k]) for k in ("Q", "K", "V", "O", "dO", "LSE", "dQ", "dK", "dV")),
                            a["B"], a["H"], a["H_kv"], a["N"], a["d"], a["scale"], a["causal"],
                            None) == code


def test_bwd_workspace_bytes(lib):
    assert ea.attn_bwd_workspace_bytes(2, 3, 300, 64) == 2 * 2 * 3 * 384 * 4
    assert ea.attn_bwd_workspace_bytes(2, 3, 300, 96) == 0
