"""Host-side pieces of bench.py (no GPU): the roofline arithmetic against the
workload figures it is quoted on, the max-over-ranks timing with two gloo
ranks, and the reference arm's JSON line on a tiny CPU sample."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

import bench
from exact_attention_tma_gb300.inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_flops_and_bytes():
    # W = 4*B*H*N^2*d (halved when causal), Q = Q,K,V read + O written + fp32 LSE.
    f, b = bench.fwd_work(WORKLOADS["causal_fwd"])
    assert f == pytest.approx(0.5 * 4 * 4 * 16 * 2048 ** 2 * 128)
    assert b == 134_742_016
    f, b = bench.fwd_work(WORKLOADS["noncausal_fwd"])
    assert f == pytest.approx(4 * 8 * 32 * 4096 ** 2 * 64)
    assert b == 541_065_216
    f, b = bench.fwd_work(WORKLOADS["long_causal_fwd"])
    assert b == 538_968_064
    f, b = bench.dec_work(WORKLOADS["decode"])
    assert f == pytest.approx(4 * 16 * 32 * 8192 * 128)
    assert b == 2_147_745_792
    # Grouped-query: K and V have h_kv = 8 heads for h = 64 query heads.
    f, b = bench.fwd_work(WORKLOADS["gqa_fwd"])
    assert f == pytest.approx(0.5 * 4 * 4 * 64 * 2048 ** 2 * 128)
    assert b == 2 * (4 * 64 * 2048 * 128) * 2 + 2 * (4 * 8 * 2048 * 128) * 2 + 4 * 64 * 2048 * 4
    f, b = bench.dec_work(WORKLOADS["gqa_decode"])
    assert f == pytest.approx(4 * 16 * 64 * 8192 * 128)
    assert b == 2 * 16 * 8 * 8192 * 128 * 2 + 2 * 16 * 64 * 128 * 2
    # Backward: five N x N x d products per head (2.5x the forward), causal
    # halved; Q, O, dO, dQ and K, V, dK, dV once each, plus the fp32 LSE.
    f, b = bench.bwd_work(WORKLOADS["causal_bwd"])
    assert f == pytest.approx(2.5 * bench.fwd_work(WORKLOADS["causal_fwd"])[0])
    assert b == 8 * (4 * 16 * 2048 * 128) * 2 + 4 * 16 * 2048 * 4


def test_roofline_time_takes_the_slower_roof():
    peaks = {"bf16_tflops": 1000.0, "hbm_gbs": 1000.0}
    assert bench.roof_time(2e12, 1e9, peaks) == pytest.approx(2e-3)   # compute-bound
    assert bench.roof_time(1e9, 3e9, peaks) == pytest.approx(3e-3)    # memory-bound
    assert bench.pct_of_roofline(1.0, 2.0) == pytest.approx(50.0)


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(1.5 + rank, world)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_prints_one_json_line():
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
           "--warmup", "3", "--cpu-fwd-heads", "1", "--cpu-dec-heads", "2"]
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["metric"] == bench.METRIC
    assert rec["unit"] == bench.UNIT and rec["higher_is_better"] is True
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["value"] == rec["value"]
