"""Seeded synthetic inputs for the attention workloads.

This module draws random numbers and nothing else: it holds none of the
attention arithmetic, so both the CUDA path and the fp64 oracle can take
their inputs from it.  Inputs are drawn in fp32 from one CPU
``torch.Generator`` seeded per workload, in the order Q, K, V (decode: q, K,
V), then rounded to bf16 with torch's round-to-nearest-even.  The oracle reads
those bf16 values (exact in fp64), so parity errors measure the kernels only.

The named workloads are the five shapes the attention path is specified on:
a tiny non-causal forward, a causal forward, a non-causal forward with peaky
scores and uniform V, a long-sequence causal forward and a split-KV decode
against a long cache.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str            # "fwd" or "decode"
    B: int
    H: int
    N: int               # sequence length (fwd) or cache length L (decode)
    d: int
    causal: bool
    seed: int
    qk_std: float = 1.0  # Q and K are N(0, qk_std^2)
    v_dist: str = "normal"   # "normal": N(0,1); "uniform": U(-1, 1)
    nsplit: int = 0      # decode only: KV split slots per head (calls use at most this many)
    scale: float = field(default=0.0)
    H_kv: int = 0        # K/V heads (grouped-query attention); 0 means H_kv = H
    page_size: int = 0   # paged decode only: tokens per page

    def __post_init__(self):
        if self.scale == 0.0:
            object.__setattr__(self, "scale", 1.0 / math.sqrt(self.d))
        if self.H_kv == 0:
            object.__setattr__(self, "H_kv", self.H)


WORKLOADS = {
    "tiny_fwd": Workload("tiny_fwd", "fwd", 1, 2, 256, 64, False, 0),
    "causal_fwd": Workload("causal_fwd", "fwd", 4, 16, 2048, 128, True, 1),
    "noncausal_fwd": Workload("noncausal_fwd", "fwd", 8, 32, 4096, 64, False, 2,
                              qk_std=1.5, v_dist="uniform"),
    "long_causal_fwd": Workload("long_causal_fwd", "fwd", 1, 32, 16384, 128, True, 3),
    "decode": Workload("decode", "decode", 16, 32, 8192, 128, False, 4, nsplit=32),
    # Grouped-query shapes (h = 64 query heads over h_kv = 8 K/V heads, g = 8, the
    # example on the pages), forward and decode.
    "gqa_fwd": Workload("gqa_fwd", "fwd", 4, 64, 2048, 128, True, 5, H_kv=8),
    "gqa_decode": Workload("gqa_decode", "decode", 16, 64, 8192, 128, False, 6, nsplit=32,
                           H_kv=8),
    # The decode workload's cache in pages of 64 tokens scattered over a shuffled
    # page pool (one block table per sequence, all sequences full length).
    "paged_decode": Workload("paged_decode", "paged", 16, 32, 8192, 128, False, 7, nsplit=32,
                             page_size=64),
    # The grouped-query decode shape on a paged cache (64-token pages).
    "paged_gqa_decode": Workload("paged_gqa_decode", "paged", 16, 64, 8192, 128, False, 12,
                                 nsplit=32, H_kv=8, page_size=64),
    # Backward of the causal forward shape: Q, K, V as the forward draws them,
    # then the upstream gradient dO ~ N(0, 1).
    "causal_bwd": Workload("causal_bwd", "bwd", 4, 16, 2048, 128, True, 8),
    # FP8 (E4M3) forward: the causal forward shapes with inputs drawn as for
    # the bf16 forward and quantised per tensor (amax / 448 scaling).
    "fp8_causal_fwd": Workload("fp8_causal_fwd", "fp8", 4, 16, 2048, 128, True, 9),
    "fp8_long_causal_fwd": Workload("fp8_long_causal_fwd", "fp8", 1, 32, 16384, 128, True, 10),
}


def _draw(gen: torch.Generator, shape, std: float, dist: str) -> torch.Tensor:
    if dist == "normal":
        x = torch.randn(shape, generator=gen, dtype=torch.float32)
        if std != 1.0:
            x = x * std
        return x
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2.0 - 1.0
    raise ValueError(f"unknown distribution {dist!r}")


def fwd_inputs(B: int, H: int, N: int, d: int, seed: int, qk_std: float = 1.0,
               v_dist: str = "normal", device="cpu", H_kv: int | None = None):
    """Q [B, H, N, d] and K, V [B, H_kv, N, d] (H_kv defaults to H), bf16 on ``device``."""
    H_kv = H if H_kv is None else H_kv
    gen = torch.Generator(device="cpu").manual_seed(seed)
    q = _draw(gen, (B, H, N, d), qk_std, "normal").to(torch.bfloat16)
    k = _draw(gen, (B, H_kv, N, d), qk_std, "normal").to(torch.bfloat16)
    v = _draw(gen, (B, H_kv, N, d), 1.0, v_dist).to(torch.bfloat16)
    return q.to(device), k.to(device), v.to(device)


def decode_inputs(B: int, H: int, L: int, d: int, seed: int, device="cpu",
                  H_kv: int | None = None):
    """q [B, H, d] and Kcache, Vcache [B, H_kv, L, d] (H_kv defaults to H), bf16."""
    H_kv = H if H_kv is None else H_kv
    gen = torch.Generator(device="cpu").manual_seed(seed)
    q = _draw(gen, (B, H, d), 1.0, "normal").to(torch.bfloat16)
    k = _draw(gen, (B, H_kv, L, d), 1.0, "normal").to(torch.bfloat16)
    v = _draw(gen, (B, H_kv, L, d), 1.0, "normal").to(torch.bfloat16)
    return q.to(device), k.to(device), v.to(device)


def paged_decode_inputs(B: int, H: int, L: int, d: int, page_size: int, seed: int, device="cpu",
                        H_kv: int | None = None, seq_lens=None, extra_pages: int = 0):
    """q [B, H, d], K/V pages [num_pages, H_kv, page_size, d] (bf16), block table
    [B, ceil(L / page_size)] and seq_lens [B] (int32).

    Pages are drawn in fp32 like the contiguous caches (q, then K pages, then V
    pages, all pages including unused ones), then a random permutation of the
    page pool (from the same generator) assigns pages to the sequences' blocks.
    """
    H_kv = H if H_kv is None else H_kv
    max_blocks = -(-L // page_size)
    num_pages = B * max_blocks + extra_pages
    gen = torch.Generator(device="cpu").manual_seed(seed)
    q = _draw(gen, (B, H, d), 1.0, "normal").to(torch.bfloat16)
    kp = _draw(gen, (num_pages, H_kv, page_size, d), 1.0, "normal").to(torch.bfloat16)
    vp = _draw(gen, (num_pages, H_kv, page_size, d), 1.0, "normal").to(torch.bfloat16)
    perm = torch.randperm(num_pages, generator=gen)[: B * max_blocks]
    table = perm.reshape(B, max_blocks).to(torch.int32)
    lens = torch.full((B,), L, dtype=torch.int32) if seq_lens is None else \
        torch.as_tensor(seq_lens, dtype=torch.int32)
    return (q.to(device), kp.to(device), vp.to(device), table.to(device), lens.to(device))


def bwd_inputs(B: int, H: int, N: int, d: int, seed: int, qk_std: float = 1.0,
               v_dist: str = "normal", device="cpu", H_kv: int | None = None):
    """Q, K, V as fwd_inputs draws them, then dO [B, H, N, d] ~ N(0, 1), bf16."""
    H_kv = H if H_kv is None else H_kv
    gen = torch.Generator(device="cpu").manual_seed(seed)
    q = _draw(gen, (B, H, N, d), qk_std, "normal").to(torch.bfloat16)
    k = _draw(gen, (B, H_kv, N, d), qk_std, "normal").to(torch.bfloat16)
    v = _draw(gen, (B, H_kv, N, d), 1.0, v_dist).to(torch.bfloat16)
    do = _draw(gen, (B, H, N, d), 1.0, "normal").to(torch.bfloat16)
    return q.to(device), k.to(device), v.to(device), do.to(device)


def fp8_inputs(B: int, H: int, N: int, d: int, seed: int, device="cpu"):
    """Q, K, V drawn as fwd_inputs draws them (fp32 N(0, 1), same order), then
    each quantised to E4M3 with one descale factor per tensor, amax / 448
    (the largest E4M3 value): code = round_to_nearest_even(x / descale).
    Returns (Q8, K8, V8) as float8_e4m3fn tensors and (descale_q, descale_k,
    descale_v)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    xs = [_draw(gen, (B, H, N, d), 1.0, "normal") for _ in range(3)]
    codes, descales = [], []
    for x in xs:
        ds = float(x.abs().max()) / 448.0
        codes.append((x / ds).to(torch.float8_e4m3fn).to(device))
        descales.append(ds)
    return tuple(codes), tuple(descales)


def workload_inputs(w: Workload, device="cpu"):
    if w.kind == "fp8":
        return fp8_inputs(w.B, w.H, w.N, w.d, w.seed, device)
    if w.kind == "bwd":
        return bwd_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_std, w.v_dist, device, w.H_kv)
    if w.kind == "fwd":
        return fwd_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_std, w.v_dist, device, w.H_kv)
    if w.kind == "paged":
        return paged_decode_inputs(w.B, w.H, w.N, w.d, w.page_size, w.seed, device, w.H_kv)
    return decode_inputs(w.B, w.H, w.N, w.d, w.seed, device, w.H_kv)
