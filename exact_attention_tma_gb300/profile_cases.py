"""Run one attention case a few times through the C ABI, for profilers.

    python -m exact_attention_tma_gb300.profile_cases --case fwd-causal --iters 3
    python -m exact_attention_tma_gb300.profile_cases --case decode --batch 4 --iters 3
    python -m exact_attention_tma_gb300.profile_cases --case gqa-decode --batch 4 --iters 3
    python -m exact_attention_tma_gb300.profile_cases --case bwd-causal --batch 1 --iters 3

Cases use the same shapes and seeded inputs as the bench workloads; decode
can be run at a smaller batch so that a multi-pass Nsight Compute capture
stays small (each head is an independent unit of work, so DRAM traffic
scales with the batch).  Inputs are generated on the device (torch RNG), since
only the kernels' behaviour is profiled here, not their values.
"""
from __future__ import annotations

import argparse

import torch

import exact_attention_tma_gb300 as ea
from exact_attention_tma_gb300.inputs import WORKLOADS

CASES = {"fwd-causal": "causal_fwd", "fwd-noncausal": "noncausal_fwd",
         "fwd-long-causal": "long_causal_fwd", "decode": "decode", "gqa-decode": "gqa_decode",
         "paged-decode": "paged_decode", "bwd-causal": "causal_bwd",
         "fp8-causal": "fp8_causal_fwd", "fp8-long-causal": "fp8_long_causal_fwd"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=sorted(CASES), required=True)
    ap.add_argument("--batch", type=int, default=0, help="override B (0 = workload's)")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    w = WORKLOADS[CASES[args.case]]
    B = args.batch or w.B
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev).manual_seed(w.seed)
    def randn(*shape):
        return torch.randn(shape, generator=g, device=dev).to(torch.bfloat16)

    if w.kind == "fp8":
        shape = (B, w.H, w.N, w.d)
        q8, k8, v8 = (randn(*shape).float().clamp(-4, 4).to(torch.float8_e4m3fn)
                      for _ in range(3))
        o = torch.empty(shape, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(shape[:3], dtype=torch.float32, device=dev)
        call = lambda: ea.attn_fwd_fp8(q8, k8, v8, o, lse, w.causal, w.scale,  # noqa: E731
                                       1.0, 1.0, 1.0)
    elif w.kind == "fwd":
        shape = (B, w.H, w.N, w.d)
        q, k, v = (randn(*shape) for _ in range(3))
        o = torch.empty_like(q)
        lse = torch.empty(shape[:3], dtype=torch.float32, device=dev)
        call = lambda: ea.attn_fwd(q, k, v, o, lse, w.causal, w.scale)  # noqa: E731
    elif w.kind == "bwd":
        q, do = randn(B, w.H, w.N, w.d), randn(B, w.H, w.N, w.d)
        k, v = randn(B, w.H_kv, w.N, w.d), randn(B, w.H_kv, w.N, w.d)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        ea.attn_fwd_gqa(q, k, v, o, lse, w.causal, w.scale)
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
        call = lambda: ea.attn_bwd(q, k, v, o, do, lse, *grads, w.causal, w.scale)  # noqa: E731
    elif w.kind == "paged":
        from exact_attention_tma_gb300.inputs import paged_decode_inputs

        ins = paged_decode_inputs(B, w.H, w.N, w.d, w.page_size, w.seed, dev, w.H_kv)
        o = torch.empty_like(ins[0])
        call = lambda: ea.attn_decode_paged(*ins, o, w.scale)  # noqa: E731
    else:
        q = randn(B, w.H, w.d)
        kc, vc = randn(B, w.H_kv, w.N, w.d), randn(B, w.H_kv, w.N, w.d)
        o = torch.empty_like(q)
        call = lambda: ea.attn_decode_gqa(q, kc, vc, o, w.scale)  # noqa: E731
    for _ in range(args.iters):
        call()
    torch.cuda.synchronize()
    status = ea.attn_get_device_status()
    if status != 0:
        raise SystemExit(f"device status {status}: {ea.attn_status_string(status)}")
    print(f"{args.case} B={B}: {args.iters} launches ok")


if __name__ == "__main__":
    main()
