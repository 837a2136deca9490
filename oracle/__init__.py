"""fp64 CPU oracle for exact attention (ctypes wrapper over attn_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product library (``exact_attention_tma_gb300``) never imports it, and this
package imports nothing from the product.

The arithmetic lives in ``attn_oracle.c`` (plain loops, fp64, single-threaded
per head; S and P materialised).  This wrapper only marshals numpy arrays and,
for many heads, runs independent per-head calls on a thread pool (ctypes drops
the GIL during each call, so heads run in parallel on the host cores).

Definition followed: "Why Fast GPUs Still Wait for Memory", section
"Attention from first principles" (S = QK^T, P = softmax(S), O = PV), with the
readings on scale, causal alignment, LSE and split-KV stated in the C file.
Every function here is pinned by ``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_long)


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into liboracle.so with gcc (no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_attention.argtypes = [
                _dp, ctypes.c_long, _dp, _dp, ctypes.c_long, ctypes.c_long,
                ctypes.c_double, ctypes.c_int, _lp, ctypes.c_long,
                _dp, _dp, _dp, _dp,
            ]
            lib.oracle_decode.argtypes = [
                _dp, _dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_double, _dp, _dp,
            ]
            lib.oracle_decode_split.argtypes = [
                _dp, _dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                ctypes.c_long, _dp, _dp,
            ]
            lib.oracle_lse_combine.argtypes = [
                _dp, _dp, ctypes.c_long, ctypes.c_long, _dp, _dp,
            ]
            lib.oracle_attention_backward.argtypes = [
                _dp, _dp, _dp, _dp, ctypes.c_long, ctypes.c_long, ctypes.c_double,
                ctypes.c_int, _dp, _dp, _dp,
            ]
            for fn in (lib.oracle_attention, lib.oracle_decode,
                       lib.oracle_decode_split, lib.oracle_lse_combine,
                       lib.oracle_attention_backward):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise RuntimeError(f"{what} failed with oracle status {rc}")


def attention_head(Q, K, V, scale: float, causal: bool, rows=None,
                   return_p: bool = False):
    """One head: Q (nq,d), K/V (nk,d).  Returns (O, LSE[, P, rowsum_err]).

    ``rows`` selects query rows (default: all).  P is (len(rows), nk).
    """
    lib = _load()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    nq, d = Q.shape
    nk = K.shape[0]
    if rows is None:
        rows_arr = None
        nrows = nq
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.shape[0]
    O = np.empty((nrows, d), np.float64)
    LSE = np.empty((nrows,), np.float64)
    P = np.empty((nrows, nk), np.float64) if return_p else None
    err = ctypes.c_double(0.0)
    rc = lib.oracle_attention(
        _ptr(Q), nq, _ptr(K), _ptr(V), nk, d, float(scale), int(bool(causal)),
        rows_arr.ctypes.data_as(_lp) if rows_arr is not None else None, nrows,
        _ptr(O), _ptr(LSE), _ptr(P) if P is not None else None, ctypes.byref(err),
    )
    _check(rc, "oracle_attention")
    if return_p:
        return O, LSE, P, err.value
    return O, LSE


def attention(Q, K, V, scale: float, causal: bool, rows=None, heads=None,
              threads: int | None = None):
    """Batched heads: Q/K/V (..., N, d).  Returns O (..., R, d), LSE (..., R).

    ``heads`` optionally lists flat head indices (over the leading dims) to
    compute; the result then has shape (len(heads), R, d).  ``rows`` selects
    query rows for every head.  Heads run on ``threads`` host threads.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    lead = Q.shape[:-2]
    N, d = Q.shape[-2:]
    Qf = Q.reshape(-1, N, d)
    Kf = K.reshape(-1, K.shape[-2], d)
    Vf = V.reshape(-1, V.shape[-2], d)
    hs = list(range(Qf.shape[0])) if heads is None else list(heads)
    R = N if rows is None else len(rows)
    O = np.empty((len(hs), R, d), np.float64)
    LSE = np.empty((len(hs), R), np.float64)

    def one(t):
        h = hs[t]
        O[t], LSE[t] = attention_head(Qf[h], Kf[h], Vf[h], scale, causal, rows)

    _run(one, len(hs), threads)
    if heads is None:
        return O.reshape(*lead, R, d), LSE.reshape(*lead, R)
    return O, LSE


def decode(q, K, V, scale: float, heads=None, threads: int | None = None):
    """Decode: q (..., d), K/V (..., L, d).  Returns O (..., d), LSE (...)."""
    lib = _load()
    q, K, V = _f64(q), _f64(K), _f64(V)
    lead = q.shape[:-1]
    d = q.shape[-1]
    L = K.shape[-2]
    qf = q.reshape(-1, d)
    Kf = K.reshape(-1, L, d)
    Vf = V.reshape(-1, L, d)
    hs = list(range(qf.shape[0])) if heads is None else list(heads)
    O = np.empty((len(hs), d), np.float64)
    LSE = np.empty((len(hs),), np.float64)

    def one(t):
        h = hs[t]
        o = np.empty((d,), np.float64)
        lse = np.empty((1,), np.float64)
        rc = lib.oracle_decode(_ptr(qf[h]), _ptr(Kf[h]), _ptr(Vf[h]), L, d,
                               float(scale), _ptr(o), _ptr(lse))
        _check(rc, "oracle_decode")
        O[t], LSE[t] = o, lse[0]

    _run(one, len(hs), threads)
    if heads is None:
        return O.reshape(*lead, d), LSE.reshape(lead)
    return O, LSE


def decode_split(q, K, V, scale: float, nsplit: int):
    """One head's split-KV partials: returns O_s (nsplit, d), lse_s (nsplit)."""
    lib = _load()
    q, K, V = _f64(q), _f64(K), _f64(V)
    L, d = K.shape
    O_s = np.empty((nsplit, d), np.float64)
    lse_s = np.empty((nsplit,), np.float64)
    rc = lib.oracle_decode_split(_ptr(q), _ptr(K), _ptr(V), L, d, float(scale),
                                 nsplit, _ptr(O_s), _ptr(lse_s))
    _check(rc, "oracle_decode_split")
    return O_s, lse_s


def lse_combine(O_s, lse_s):
    """Combine normalised partials: returns O (d), LSE (scalar)."""
    lib = _load()
    O_s, lse_s = _f64(O_s), _f64(lse_s)
    nsplit, d = O_s.shape
    O = np.empty((d,), np.float64)
    lse = np.empty((1,), np.float64)
    rc = lib.oracle_lse_combine(_ptr(O_s), _ptr(lse_s), nsplit, d, _ptr(O), _ptr(lse))
    _check(rc, "oracle_lse_combine")
    return O, lse[0]


def kv_head_of(h: int, H: int, H_kv: int) -> int:
    """K/V head that query head h reads under grouped-query attention.

    "Why Fast GPUs Still Wait for Memory", section "Attention III · KV cache,
    GQA, MLA": h query heads share h_kv key/value heads with group size
    g = h / h_kv (MQA is g = h).  Reading: the groups are contiguous, so query
    head h uses K/V head floor(h / g).
    """
    if H_kv < 1 or H % H_kv != 0 or not 0 <= h < H:
        raise ValueError("need 1 <= H_kv, H % H_kv == 0 and 0 <= h < H")
    return h // (H // H_kv)


def attention_gqa(Q, K, V, scale: float, causal: bool, rows=None, heads=None,
                  threads: int | None = None):
    """Grouped-query forward: Q (B, H, N, d), K/V (B, H_kv, N, d).

    Every (b, h) is one call of the per-head definition with K/V head
    ``kv_head_of(h)``.  ``heads`` optionally lists flat (b * H + h) indices.
    Returns O (B, H, R, d), LSE (B, H, R), or (len(heads), R, d) / (len(heads), R).
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, d = Q.shape
    H_kv = K.shape[1]
    hs = list(range(B * H)) if heads is None else list(heads)
    R = N if rows is None else len(rows)
    O = np.empty((len(hs), R, d), np.float64)
    LSE = np.empty((len(hs), R), np.float64)

    def one(t):
        b, h = divmod(hs[t], H)
        kh = kv_head_of(h, H, H_kv)
        O[t], LSE[t] = attention_head(Q[b, h], K[b, kh], V[b, kh], scale, causal, rows)

    _run(one, len(hs), threads)
    if heads is None:
        return O.reshape(B, H, R, d), LSE.reshape(B, H, R)
    return O, LSE


def decode_gqa(q, K, V, scale: float, heads=None, threads: int | None = None):
    """Grouped-query decode: q (B, H, d), K/V (B, H_kv, L, d).

    Returns O (B, H, d), LSE (B, H), or per listed flat head.
    """
    lib = _load()
    q, K, V = _f64(q), _f64(K), _f64(V)
    B, H, d = q.shape
    H_kv, L = K.shape[1], K.shape[2]
    hs = list(range(B * H)) if heads is None else list(heads)
    O = np.empty((len(hs), d), np.float64)
    LSE = np.empty((len(hs),), np.float64)

    def one(t):
        b, h = divmod(hs[t], H)
        kh = kv_head_of(h, H, H_kv)
        Kh, Vh = np.ascontiguousarray(K[b, kh]), np.ascontiguousarray(V[b, kh])
        qh = np.ascontiguousarray(q[b, h])
        o = np.empty((d,), np.float64)
        lse = np.empty((1,), np.float64)
        rc = lib.oracle_decode(_ptr(qh), _ptr(Kh), _ptr(Vh), L, d, float(scale), _ptr(o),
                               _ptr(lse))
        _check(rc, "oracle_decode")
        O[t], LSE[t] = o, lse[0]

    _run(one, len(hs), threads)
    if heads is None:
        return O.reshape(B, H, d), LSE.reshape(B, H)
    return O, LSE


def paged_rows(pages, block_table_row, seq_len: int, kv_head: int):
    """The first ``seq_len`` K (or V) rows of one sequence from a paged cache.

    "M4.2 - GPU Execution Model for Transformer Kernels" (pitfall 16 and the
    kernel contract of its coalescing section): logical K/V continuity does
    not imply contiguous physical addresses; the decode walks the page/block
    layout.  Reading: ``pages`` is (num_pages, H_kv, page_size, d), logical
    token t of the sequence lives in page ``block_table_row[t // page_size]``
    at slot ``t % page_size``.
    """
    page_size = pages.shape[2]
    t = np.arange(seq_len)
    ids = np.asarray(block_table_row)[t // page_size]
    return pages[ids, kv_head, t % page_size]


def decode_paged(q, K_pages, V_pages, block_table, seq_lens, scale: float, heads=None,
                 threads: int | None = None):
    """Paged (and grouped-query) decode: q (B, H, d); K/V pages
    (num_pages, H_kv, page_size, d); block_table (B, max_blocks) page ids;
    seq_lens (B).  Query head h reads K/V head ``kv_head_of(h)`` over the
    sequence's first seq_lens[b] tokens.  Returns O (B, H, d), LSE (B, H), or
    per listed flat head.
    """
    lib = _load()
    q, Kp, Vp = _f64(q), _f64(K_pages), _f64(V_pages)
    B, H, d = q.shape
    H_kv = Kp.shape[1]
    hs = list(range(B * H)) if heads is None else list(heads)
    O = np.empty((len(hs), d), np.float64)
    LSE = np.empty((len(hs),), np.float64)

    def one(t):
        b, h = divmod(hs[t], H)
        kh = kv_head_of(h, H, H_kv)
        L = int(seq_lens[b])
        Kh = np.ascontiguousarray(paged_rows(Kp, block_table[b], L, kh))
        Vh = np.ascontiguousarray(paged_rows(Vp, block_table[b], L, kh))
        qh = np.ascontiguousarray(q[b, h])
        o = np.empty((d,), np.float64)
        lse = np.empty((1,), np.float64)
        rc = lib.oracle_decode(_ptr(qh), _ptr(Kh), _ptr(Vh), L, d, float(scale), _ptr(o),
                               _ptr(lse))
        _check(rc, "oracle_decode")
        O[t], LSE[t] = o, lse[0]

    _run(one, len(hs), threads)
    if heads is None:
        return O.reshape(B, H, d), LSE.reshape(B, H)
    return O, LSE


def attention_backward_head(Q, K, V, dO, scale: float, causal: bool):
    """Gradients of one head: Q, K, V, dO (n, d).  Returns (dQ, dK, dV).

    The chain rule through S = scale QK^T (masked), P = softmax(S), O = PV,
    with S and P materialised ("Why Fast GPUs Still Wait for Memory",
    "FlashAttention is an IO algorithm": the backward pass recomputes S).
    """
    lib = _load()
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    n, d = Q.shape
    dQ = np.empty((n, d), np.float64)
    dK = np.empty((n, d), np.float64)
    dV = np.empty((n, d), np.float64)
    rc = lib.oracle_attention_backward(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), n, d, float(scale),
                                       int(bool(causal)), _ptr(dQ), _ptr(dK), _ptr(dV))
    _check(rc, "oracle_attention_backward")
    return dQ, dK, dV


def attention_backward(Q, K, V, dO, scale: float, causal: bool, heads=None,
                       threads: int | None = None):
    """Batched gradients: Q, dO (B, H, N, d); K, V (B, H_kv, N, d) with
    H % H_kv == 0 (H_kv = H is plain multi-head attention).

    Returns dQ (B, H, N, d) and dK, dV (B, H_kv, N, d): under grouped-query
    attention a K/V head's gradient is the sum over the query heads that read
    it (query head h reads K/V head kv_head_of(h)).  With ``heads`` (flat
    query-head indices) only those heads are computed and the per-query-head
    gradients are returned unsummed, each of shape (len(heads), N, d).
    """
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, d = Q.shape
    H_kv = K.shape[1]
    if H % H_kv:
        raise ValueError("H must be a multiple of H_kv")
    hs = list(range(B * H)) if heads is None else list(heads)
    dQh = np.empty((len(hs), N, d), np.float64)
    dKh = np.empty((len(hs), N, d), np.float64)
    dVh = np.empty((len(hs), N, d), np.float64)

    def one(t):
        b, h = divmod(hs[t], H)
        kh = kv_head_of(h, H, H_kv)
        dQh[t], dKh[t], dVh[t] = attention_backward_head(Q[b, h], K[b, kh], V[b, kh], dO[b, h],
                                                         scale, causal)

    _run(one, len(hs), threads)
    if heads is not None:
        return dQh, dKh, dVh
    dK = np.zeros((B, H_kv, N, d), np.float64)
    dV = np.zeros((B, H_kv, N, d), np.float64)
    for t, flat in enumerate(hs):
        b, h = divmod(flat, H)
        kh = kv_head_of(h, H, H_kv)
        dK[b, kh] += dKh[t]
        dV[b, kh] += dVh[t]
    return dQh.reshape(B, H, N, d), dK, dV


def e4m3_value(code: int) -> float:
    """Value of one 8-bit E4M3 code (the "fn" encoding the tensor cores read
    as e4m3): bit 7 sign, bits 6-3 exponent with bias 7, bits 2-0 mantissa.
    Exponent field 0 is subnormal, value = mantissa/8 * 2^-6; codes 0x7F and
    0xFF are NaN; there are no infinities (the largest finite value is 448)."""
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    mant = code & 0x7
    if e == 0xF and mant == 0x7:
        return float("nan")
    if e == 0:
        return sign * (mant / 8.0) * 2.0 ** -6
    return sign * (1.0 + mant / 8.0) * 2.0 ** (e - 7)


_E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def decode_e4m3(codes) -> np.ndarray:
    """Exact fp64 values of an array of E4M3 codes (uint8)."""
    return _E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def attention_fp8(Q8, K8, V8, descale_q: float, descale_k: float, descale_v: float,
                  scale: float, causal: bool, rows=None, heads=None, threads: int | None = None):
    """Attention of FP8 inputs: each E4M3 code array (..., N, d) is decoded
    exactly and multiplied by its tensor's descale factor, then the plain
    definition (``attention``) runs on those fp64 values.  Returns O, LSE."""
    Q = decode_e4m3(Q8) * float(descale_q)
    K = decode_e4m3(K8) * float(descale_k)
    V = decode_e4m3(V8) * float(descale_v)
    return attention(Q, K, V, scale, causal, rows=rows, heads=heads, threads=threads)


def _run(fn, n: int, threads: int | None) -> None:
    if n == 0:
        return
    threads = threads or min(n, os.cpu_count() or 1)
    if threads <= 1 or n == 1:
        for t in range(n):
            fn(t)
        return
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(fn, range(n)))
