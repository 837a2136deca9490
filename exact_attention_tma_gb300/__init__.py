"""GB300-native exact attention: Python binding of the C ABI in include/exact_attn.h.

Every function here only marshals arguments (checks dtypes, shapes and
contiguity, passes device pointers and the CUDA stream handle) and calls the
same-named entry point of ``lib/libexact_attn.so``; all arithmetic runs in the
library's sm_103a kernels.  There is no CPU fallback: if the library is not
built, the first call raises.  Build it with ``python -m
exact_attention_tma_gb300.build`` (or ``__graft_entry__.build()``).

PyTorch is used only to hold device memory and to name the stream.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "AttnError", "attn_fwd", "attn_decode", "attn_decode_ws",
    "attn_decode_workspace_bytes", "attn_get_device_status", "attn_status_string",
    "attn_decode_num_splits", "attn_decode_noalloc", "attn_selftest_bounded_wait", "forward",
    "decode", "library_path", "load",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "lib", "libexact_attn.so")
_lib = None
_lock = threading.Lock()

# attn_status codes (include/exact_attn.h)
(ATTN_OK, ATTN_ERR_NULL, ATTN_ERR_SHAPE, ATTN_ERR_HEADDIM, ATTN_ERR_ALIGN, ATTN_ERR_CUDA,
 ATTN_ERR_NOMEM, ATTN_ERR_TIMEOUT, ATTN_ERR_ARG) = range(9)


class AttnError(RuntimeError):
    """A non-OK attn_status returned by the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {attn_status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libexact_attn.so (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    f"CUDA library {_LIB_PATH} is missing; build it with "
                    "`python -m exact_attention_tma_gb300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
            lib.attn_decode.argtypes = [vp, vp, vp, vp, i, i, i, i, f, vp]
            lib.attn_decode_ws.argtypes = [vp, vp, vp, vp, i, i, i, i, f, vp, sz, vp]
            lib.attn_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
            lib.attn_decode_gqa.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp]
            lib.attn_decode_gqa_ws.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
            lib.attn_decode_paged.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
            lib.attn_fwd_fp8.argtypes = [vp] * 5 + [i, i, i, i, f, f, f, f, i, vp]
            lib.attn_fwd_fp8_ws.argtypes = [vp] * 5 + [i, i, i, i, f, f, f, f, i, vp, sz, vp]
            lib.attn_fwd_fp8_workspace_bytes.argtypes = [i, i, i, i]
            lib.attn_fwd_fp8_workspace_bytes.restype = sz
            lib.attn_bwd.argtypes = [vp] * 9 + [i, i, i, i, f, i, vp]
            lib.attn_bwd_gqa.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, vp]
            lib.attn_bwd_gqa_ws.argtypes = [vp] * 9 + [i, i, i, i, i, f, i, vp, sz, vp]
            lib.attn_bwd_workspace_bytes.argtypes = [i, i, i, i]
            lib.attn_bwd_workspace_bytes.restype = sz
            lib.attn_selftest_bounded_wait.argtypes = [i, vp]
            lib.attn_selftest_bounded_wait.restype = ctypes.c_int
            lib.attn_decode_noalloc.argtypes = [vp, vp, vp, vp, i, i, i, i, f, vp]
            lib.attn_decode_noalloc.restype = ctypes.c_int
            lib.attn_decode_workspace_bytes.argtypes = [i, i, i, i]
            lib.attn_decode_workspace_bytes.restype = sz
            lib.attn_get_device_status.argtypes = [vp]
            lib.attn_status_string.argtypes = [i]
            lib.attn_status_string.restype = ctypes.c_char_p
            lib.attn_decode_num_splits.argtypes = []
            for fn in (lib.attn_fwd, lib.attn_decode, lib.attn_decode_ws, lib.attn_fwd_gqa,
                       lib.attn_decode_gqa, lib.attn_decode_gqa_ws, lib.attn_decode_paged,
                       lib.attn_get_device_status, lib.attn_decode_num_splits, lib.attn_bwd,
                       lib.attn_bwd_gqa, lib.attn_bwd_gqa_ws, lib.attn_fwd_fp8,
                       lib.attn_fwd_fp8_ws):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _stream(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t, name, dtype):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _check(status: int, what: str) -> None:
    if status != ATTN_OK:
        raise AttnError(status, what)


def attn_status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def attn_decode_num_splits() -> int:
    return load().attn_decode_num_splits()


def attn_fwd(Q, K, V, O, LSE, causal: bool, scale: float, stream=None) -> None:
    """O, LSE <- attention(Q, K, V); all [B, H, N, d] bf16 (LSE [B, H, N] fp32)."""
    import torch

    B, H, N, d = Q.shape
    for name, t in (("K", K), ("V", V), ("O", O)):
        if tuple(t.shape) != (B, H, N, d):
            raise ValueError(f"{name} shape {tuple(t.shape)} != Q shape {(B, H, N, d)}")
    if tuple(LSE.shape) != (B, H, N):
        raise ValueError(f"LSE shape {tuple(LSE.shape)} != {(B, H, N)}")
    args = [_dev(Q, "Q", torch.bfloat16), _dev(K, "K", torch.bfloat16),
            _dev(V, "V", torch.bfloat16), _dev(O, "O", torch.bfloat16),
            _dev(LSE, "LSE", torch.float32)]
    _check(load().attn_fwd(*args, B, H, N, d, float(scale), int(bool(causal)),
                           _stream(stream)), "attn_fwd")


def attn_fwd_gqa(Q, K, V, O, LSE, causal: bool, scale: float, stream=None) -> None:
    """Grouped-query forward: Q, O [B, H, N, d], K, V [B, H_kv, N, d] bf16, LSE [B, H, N]."""
    import torch

    B, H, N, d = Q.shape
    H_kv = K.shape[1]
    if tuple(K.shape) != (B, H_kv, N, d) or tuple(V.shape) != (B, H_kv, N, d):
        raise ValueError(f"K/V shape must be {(B, H_kv, N, d)}")
    if tuple(O.shape) != (B, H, N, d):
        raise ValueError(f"O shape {tuple(O.shape)} != Q shape {(B, H, N, d)}")
    if tuple(LSE.shape) != (B, H, N):
        raise ValueError(f"LSE shape {tuple(LSE.shape)} != {(B, H, N)}")
    args = [_dev(Q, "Q", torch.bfloat16), _dev(K, "K", torch.bfloat16),
            _dev(V, "V", torch.bfloat16), _dev(O, "O", torch.bfloat16),
            _dev(LSE, "LSE", torch.float32)]
    _check(load().attn_fwd_gqa(*args, B, H, H_kv, N, d, float(scale), int(bool(causal)),
                               _stream(stream)), "attn_fwd_gqa")


def _fp8_args(Q8, K8, V8, O, LSE):
    import torch

    B, H, N, d = Q8.shape
    for name, t in (("K8", K8), ("V8", V8)):
        if tuple(t.shape) != (B, H, N, d):
            raise ValueError(f"{name} shape {tuple(t.shape)} != {(B, H, N, d)}")
    if tuple(O.shape) != (B, H, N, d):
        raise ValueError(f"O shape {tuple(O.shape)} != {(B, H, N, d)}")
    if tuple(LSE.shape) != (B, H, N):
        raise ValueError(f"LSE shape {tuple(LSE.shape)} != {(B, H, N)}")
    f8 = torch.float8_e4m3fn
    args = [_dev(Q8, "Q8", f8), _dev(K8, "K8", f8), _dev(V8, "V8", f8),
            _dev(O, "O", torch.bfloat16), _dev(LSE, "LSE", torch.float32)]
    return args, B, H, N, d


def attn_fwd_fp8(Q8, K8, V8, O, LSE, causal: bool, scale: float, descale_q: float,
                 descale_k: float, descale_v: float, stream=None) -> None:
    """FP8 forward: Q8, K8, V8 float8_e4m3fn [B, H, N, 128] with per-tensor
    descale factors (value = code * descale); O bf16, LSE fp32 [B, H, N]."""
    args, B, H, N, d = _fp8_args(Q8, K8, V8, O, LSE)
    _check(load().attn_fwd_fp8(*args, B, H, N, d, float(scale), float(descale_q),
                               float(descale_k), float(descale_v), int(bool(causal)),
                               _stream(stream)), "attn_fwd_fp8")


def attn_fwd_fp8_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().attn_fwd_fp8_workspace_bytes(B, H, N, d))


def _bwd_args(Q, K, V, O, dO, LSE, dQ, dK, dV):
    import torch

    B, H, N, d = Q.shape
    H_kv = K.shape[1]
    for name, t in (("K", K), ("V", V), ("dK", dK), ("dV", dV)):
        if tuple(t.shape) != (B, H_kv, N, d):
            raise ValueError(f"{name} shape {tuple(t.shape)} != {(B, H_kv, N, d)}")
    for name, t in (("O", O), ("dO", dO), ("dQ", dQ)):
        if tuple(t.shape) != (B, H, N, d):
            raise ValueError(f"{name} shape {tuple(t.shape)} != {(B, H, N, d)}")
    if tuple(LSE.shape) != (B, H, N):
        raise ValueError(f"LSE shape {tuple(LSE.shape)} != {(B, H, N)}")
    args = [_dev(Q, "Q", torch.bfloat16), _dev(K, "K", torch.bfloat16),
            _dev(V, "V", torch.bfloat16), _dev(O, "O", torch.bfloat16),
            _dev(dO, "dO", torch.bfloat16), _dev(LSE, "LSE", torch.float32),
            _dev(dQ, "dQ", torch.bfloat16), _dev(dK, "dK", torch.bfloat16),
            _dev(dV, "dV", torch.bfloat16)]
    return args, B, H, H_kv, N, d


def attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, causal: bool, scale: float, stream=None) -> None:
    """Backward of attn_fwd / attn_fwd_gqa: writes dQ [B, H, N, d] and dK, dV
    [B, H_kv, N, d] (bf16) from Q, K, V, the forward's O and LSE, and dO.
    H_kv = K.shape[1] (H_kv < H: grouped-query; dK, dV sum over each group)."""
    args, B, H, H_kv, N, d = _bwd_args(Q, K, V, O, dO, LSE, dQ, dK, dV)
    _check(load().attn_bwd_gqa(*args, B, H, H_kv, N, d, float(scale), int(bool(causal)),
                               _stream(stream)), "attn_bwd_gqa")


def attn_bwd_ws(Q, K, V, O, dO, LSE, dQ, dK, dV, causal: bool, scale: float, ws,
                stream=None) -> None:
    """attn_bwd with a caller-owned workspace tensor ``ws`` (any dtype, CUDA)."""
    import torch

    args, B, H, H_kv, N, d = _bwd_args(Q, K, V, O, dO, LSE, dQ, dK, dV)
    if not (isinstance(ws, torch.Tensor) and ws.is_cuda and ws.is_contiguous()):
        raise ValueError("ws must be a contiguous CUDA tensor")
    nbytes = ws.numel() * ws.element_size()
    _check(load().attn_bwd_gqa_ws(*args, B, H, H_kv, N, d, float(scale), int(bool(causal)),
                                  ctypes.c_void_p(ws.data_ptr()), nbytes, _stream(stream)),
           "attn_bwd_gqa_ws")


def attn_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().attn_bwd_workspace_bytes(B, H, N, d))


def _gqa_decode_args(q, Kcache, Vcache, O):
    import torch

    B, H_kv, L, d = Kcache.shape
    if tuple(Vcache.shape) != (B, H_kv, L, d):
        raise ValueError("Vcache shape must match Kcache")
    if q.dim() != 3 or q.shape[0] != B or q.shape[2] != d:
        raise ValueError(f"q shape {tuple(q.shape)} must be (B, H, d) = ({B}, H, {d})")
    H = q.shape[1]
    if tuple(O.shape) != (B, H, d):
        raise ValueError(f"O shape {tuple(O.shape)} != {(B, H, d)}")
    args = [_dev(q, "q", torch.bfloat16), _dev(Kcache, "Kcache", torch.bfloat16),
            _dev(Vcache, "Vcache", torch.bfloat16), _dev(O, "O", torch.bfloat16)]
    return args, B, H, H_kv, L, d


def attn_decode_gqa(q, Kcache, Vcache, O, scale: float, stream=None) -> None:
    """Grouped-query decode: q, O [B, H, d], Kcache/Vcache [B, H_kv, L, d] bf16."""
    args, B, H, H_kv, L, d = _gqa_decode_args(q, Kcache, Vcache, O)
    _check(load().attn_decode_gqa(*args, B, H, H_kv, L, d, float(scale), _stream(stream)),
           "attn_decode_gqa")


def attn_decode_gqa_ws(q, Kcache, Vcache, O, scale: float, ws, stream=None) -> None:
    """attn_decode_gqa with a caller-owned workspace tensor ``ws`` (any dtype, CUDA)."""
    import torch

    args, B, H, H_kv, L, d = _gqa_decode_args(q, Kcache, Vcache, O)
    if not (isinstance(ws, torch.Tensor) and ws.is_cuda and ws.is_contiguous()):
        raise ValueError("ws must be a contiguous CUDA tensor")
    nbytes = ws.numel() * ws.element_size()
    _check(load().attn_decode_gqa_ws(*args, B, H, H_kv, L, d, float(scale),
                                     ctypes.c_void_p(ws.data_ptr()), nbytes, _stream(stream)),
           "attn_decode_gqa_ws")


def attn_decode_paged(q, K_pages, V_pages, block_table, seq_lens, O, scale: float,
                      stream=None) -> None:
    """Decode against a paged cache: q, O [B, H, d] bf16; K/V pages
    [num_pages, H_kv, page_size, d] bf16; block_table [B, max_blocks] int32;
    seq_lens [B] int32 (all on the GPU)."""
    import torch

    num_pages, H_kv, page_size, d = K_pages.shape
    if tuple(V_pages.shape) != tuple(K_pages.shape):
        raise ValueError("V_pages shape must match K_pages")
    if q.dim() != 3 or q.shape[2] != d:
        raise ValueError(f"q shape {tuple(q.shape)} must be (B, H, {d})")
    B, H = q.shape[0], q.shape[1]
    if tuple(O.shape) != (B, H, d):
        raise ValueError(f"O shape {tuple(O.shape)} != {(B, H, d)}")
    if block_table.dim() != 2 or block_table.shape[0] != B:
        raise ValueError("block_table must be (B, max_blocks)")
    if tuple(seq_lens.shape) != (B,):
        raise ValueError("seq_lens must be (B,)")
    max_blocks = block_table.shape[1]
    args = [_dev(q, "q", torch.bfloat16), _dev(K_pages, "K_pages", torch.bfloat16),
            _dev(V_pages, "V_pages", torch.bfloat16),
            _dev(block_table, "block_table", torch.int32), _dev(seq_lens, "seq_lens", torch.int32),
            _dev(O, "O", torch.bfloat16)]
    _check(load().attn_decode_paged(*args, B, H, H_kv, num_pages, page_size, max_blocks, d,
                                    float(scale), _stream(stream)), "attn_decode_paged")


def attn_decode(q, Kcache, Vcache, O, scale: float, stream=None) -> None:
    """O [B, H, d] <- attention of q [B, H, d] over Kcache/Vcache [B, H, L, d]."""
    import torch

    B, H, L, d = Kcache.shape
    if tuple(Vcache.shape) != (B, H, L, d):
        raise ValueError("Vcache shape must match Kcache")
    for name, t in (("q", q), ("O", O)):
        if tuple(t.shape) != (B, H, d):
            raise ValueError(f"{name} shape {tuple(t.shape)} != {(B, H, d)}")
    args = [_dev(q, "q", torch.bfloat16), _dev(Kcache, "Kcache", torch.bfloat16),
            _dev(Vcache, "Vcache", torch.bfloat16), _dev(O, "O", torch.bfloat16)]
    _check(load().attn_decode(*args, B, H, L, d, float(scale), _stream(stream)),
           "attn_decode")


def attn_decode_workspace_bytes(B: int, H: int, L: int, d: int) -> int:
    return int(load().attn_decode_workspace_bytes(B, H, L, d))


def attn_decode_ws(q, Kcache, Vcache, O, scale: float, ws, stream=None) -> None:
    """attn_decode with a caller-owned workspace tensor ``ws`` (any dtype, CUDA)."""
    import torch

    B, H, L, d = Kcache.shape
    if tuple(Vcache.shape) != (B, H, L, d):
        raise ValueError("Vcache shape must match Kcache")
    for name, t in (("q", q), ("O", O)):
        if tuple(t.shape) != (B, H, d):
            raise ValueError(f"{name} shape {tuple(t.shape)} != {(B, H, d)}")
    if not (isinstance(ws, torch.Tensor) and ws.is_cuda and ws.is_contiguous()):
        raise ValueError("ws must be a contiguous CUDA tensor")
    args = [_dev(q, "q", torch.bfloat16), _dev(Kcache, "Kcache", torch.bfloat16),
            _dev(Vcache, "Vcache", torch.bfloat16), _dev(O, "O", torch.bfloat16)]
    nbytes = ws.numel() * ws.element_size()
    _check(load().attn_decode_ws(*args, B, H, L, d, float(scale),
                                 ctypes.c_void_p(ws.data_ptr()), nbytes, _stream(stream)),
           "attn_decode_ws")


def attn_decode_noalloc(q, Kcache, Vcache, O, scale: float, stream=None) -> None:
    """attn_decode without any device allocation, for callers that cannot allocate.

    The partials go to a fixed 16 MiB scratch array inside the library (one per
    GPU, held until exit) instead of memory the library or the caller allocates;
    see include/exact_attn.h for the size limit and the sharing rules.
    """
    import torch

    B, H, L, d = Kcache.shape
    if tuple(Vcache.shape) != (B, H, L, d):
        raise ValueError("Vcache shape must match Kcache")
    for name, t in (("q", q), ("O", O)):
        if tuple(t.shape) != (B, H, d):
            raise ValueError(f"{name} shape {tuple(t.shape)} != {(B, H, d)}")
    args = [_dev(q, "q", torch.bfloat16), _dev(Kcache, "Kcache", torch.bfloat16),
            _dev(Vcache, "Vcache", torch.bfloat16), _dev(O, "O", torch.bfloat16)]
    _check(load().attn_decode_noalloc(*args, B, H, L, d, float(scale), _stream(stream)),
           "attn_decode_noalloc")


def attn_selftest_bounded_wait(limit_ms: int, stream=None) -> None:
    """Launch the bounded-wait self-test (see include/exact_attn_selftest.h)."""
    _check(load().attn_selftest_bounded_wait(int(limit_ms), _stream(stream)),
           "attn_selftest_bounded_wait")


def attn_get_device_status(stream=None) -> int:
    """Synchronise ``stream`` and return (and clear) the device status code."""
    return int(load().attn_get_device_status(_stream(stream)))


def forward(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """Allocate O and LSE on q's device and run attn_fwd.  Returns (O, LSE)."""
    import torch

    B, H, N, d = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    attn_fwd(q, k, v, o, lse, causal, d ** -0.5 if scale is None else scale, stream)
    return o, lse


def decode(q, Kcache, Vcache, scale: float | None = None, stream=None):
    """Allocate O on q's device and run attn_decode.  Returns O [B, H, d]."""
    import torch

    o = torch.empty_like(q)
    d = q.shape[-1]
    attn_decode(q, Kcache, Vcache, o, d ** -0.5 if scale is None else scale, stream)
    return o
