"""GPU parity of the fused forward kernel against the fp64 oracle.

Small shapes are compared element by element over every output (they span
several 128-row / 128-key tiles and ragged tails); the full-size workloads
are compared on sampled heads and rows that the oracle computes one by one,
in the same launch configuration the bench uses.
"""
import numpy as np
import pytest
import torch

import exact_attention_tma_gb300 as ea
from exact_attention_tma_gb300.inputs import WORKLOADS, fwd_inputs, workload_inputs
from parity import assert_within, compare_fwd, oracle_fwd, oracle_fwd_head_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from exact_attention_tma_gb300 import build

    build.build()
    ea.load()
    yield
    assert ea.attn_get_device_status() == 0


def _run(q, k, v, causal, scale):
    o, lse = ea.forward(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o, lse


def _full_check(B, H, N, d, causal, seed, qk_std=1.0, v_dist="normal"):
    q, k, v = fwd_inputs(B, H, N, d, seed, qk_std, v_dist, device="cuda")
    scale = d ** -0.5
    o, lse = _run(q, k, v, causal, scale)
    O_ref, L_ref = oracle_fwd(q, k, v, scale, causal)
    st = compare_fwd(o, lse, O_ref, L_ref, range(B * H), None)
    assert_within(st)
    return st


def test_tiny_workload_full():
    w = WORKLOADS["tiny_fwd"]
    q, k, v = workload_inputs(w, device="cuda")
    o, lse = _run(q, k, v, w.causal, w.scale)
    O_ref, L_ref = oracle_fwd(q, k, v, w.scale, w.causal)
    assert_within(compare_fwd(o, lse, O_ref, L_ref, range(w.B * w.H), None))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 300, 513])
def test_small_shapes_full(N, d, causal):
    _full_check(1, 2, N, d, causal, seed=100 + N)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_multi_head_multi_tile_full(d, causal):
    _full_check(2, 3, 1000, d, causal, seed=7)


@pytest.mark.parametrize("causal", [False, True])
def test_peaky_scores_full(causal):
    # Large score spread forces frequent running-max updates and O rescaling.
    _full_check(1, 2, 640, 64, causal, seed=9, qk_std=3.0, v_dist="uniform")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_growing_scores_force_rescales(d, causal):
    # Keys grow in norm along the sequence, so each row's running max keeps
    # jumping by more than 2^8 and the output accumulator is rescaled at many
    # K/V steps (exercises the rescale/P-buffer ordering of the pipeline).
    # V ~ U(-1, 1) keeps |O| <= 1, so bf16 rounding of P and O stays far inside
    # the tolerance even though these softmax rows are very peaky.
    B, H, N = 1, 2, 1100
    q, k, v = fwd_inputs(B, H, N, d, 77, v_dist="uniform", device="cpu")
    ramp = torch.linspace(0.2, 6.0, N).view(1, 1, N, 1)
    k = (k.float() * ramp).to(torch.bfloat16)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    scale = d ** -0.5
    o, lse = _run(q, k, v, causal, scale)
    O_ref, L_ref = oracle_fwd(q, k, v, scale, causal)
    assert_within(compare_fwd(o, lse, O_ref, L_ref, range(B * H), None))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_far_negative_scores(d, causal):
    # Every score lies far below zero (about -170 in natural-log units, with
    # unit spread): softmax is shift-invariant, so O and LSE - (common shift)
    # behave as for centred scores, but a kernel that starts its running
    # maximum at 0 sees every P underflow and must fall back to the true maximum.
    B, H, N = 1, 2, 700
    q, k, v = fwd_inputs(B, H, N, d, 91, v_dist="uniform", device="cpu")
    base = torch.full((d,), 4.0 * (128.0 / d) ** 0.5)
    q = (q.float() * 0.5 + base).to(torch.bfloat16).cuda()
    k = (k.float() * 0.5 - base).to(torch.bfloat16).cuda()
    v = v.cuda()
    scale = d ** -0.5
    o, lse = _run(q, k, v, causal, scale)
    O_ref, L_ref = oracle_fwd(q, k, v, scale, causal)
    assert L_ref.max() < -100
    assert_within(compare_fwd(o, lse, O_ref, L_ref, range(B * H), None))


def _sampled(name, heads, rows, full_heads=()):
    w = WORKLOADS[name]
    q, k, v = workload_inputs(w, device="cuda")
    o, lse = _run(q, k, v, w.causal, w.scale)
    O_ref, L_ref = oracle_fwd(q, k, v, w.scale, w.causal, heads=heads, rows=rows)
    assert_within(compare_fwd(o, lse, O_ref, L_ref, heads, rows))
    for h in full_heads:
        O_ref, L_ref = oracle_fwd(q, k, v, w.scale, w.causal, heads=[h])
        assert_within(compare_fwd(o, lse, O_ref, L_ref, [h], None))
    return o, lse


def _rows(N, n, seed):
    rng = np.random.default_rng(seed)
    edge = [0, 1, 126, 127, 128, 129, N // 2, N - 129, N - 128, N - 2, N - 1]
    return sorted(set(edge) | set(rng.choice(N, n, replace=False).tolist()))


def test_causal_workload_sampled():
    w = WORKLOADS["causal_fwd"]
    _sampled("causal_fwd", heads=range(w.B * w.H), rows=_rows(w.N, 48, 1),
             full_heads=[0, w.B * w.H - 1])


def test_noncausal_workload_sampled():
    w = WORKLOADS["noncausal_fwd"]
    heads = np.random.default_rng(2).choice(w.B * w.H, 24, replace=False).tolist()
    _sampled("noncausal_fwd", heads=sorted(heads), rows=_rows(w.N, 40, 2),
             full_heads=[5, w.B * w.H - 1])


def _one_row_per_tile(N, seed):
    """One row in every 128-row query tile (at a varying offset), plus tile edges."""
    rng = np.random.default_rng(seed)
    rows = {t * 128 + int(rng.integers(128)) for t in range(N // 128)}
    return sorted(rows | {0, 127, 128, 255, N - 129, N - 128, N - 1})


def test_long_causal_workload_sampled():
    # Every head, one row in each 128-row query tile: every persistent work
    # item of the launch (the short causal blocks of the last heads included)
    # contributes compared rows.
    w = WORKLOADS["long_causal_fwd"]
    _sampled("long_causal_fwd", heads=range(w.B * w.H), rows=_one_row_per_tile(w.N, 3))


def test_long_causal_workload_one_full_head():
    # Head 17 in full (all 16384 rows), the oracle's rows split over the host cores.
    w = WORKLOADS["long_causal_fwd"]
    q, k, v = workload_inputs(w, device="cuda")
    o, lse = _run(q, k, v, w.causal, w.scale)
    O_ref, L_ref = oracle_fwd_head_rows(q, k, v, w.scale, w.causal, 17, range(w.N))
    assert_within(compare_fwd(o, lse, O_ref, L_ref, [17], None))


@pytest.mark.parametrize("d", [64, 128])
def test_deterministic_and_no_out_of_bounds_writes(d):
    B, H, N = 2, 2, 333
    q, k, v = fwd_inputs(B, H, N, d, 21, device="cuda")
    pad = 4096
    o_buf = torch.full((B * H * N * d + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * H * N + pad,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[: B * H * N * d].view(B, H, N, d)
    lse = l_buf[: B * H * N].view(B, H, N)
    outs = []
    for _ in range(2):
        ea.attn_fwd(q, k, v, o, lse, True, d ** -0.5)
        torch.cuda.synchronize()
        outs.append((o.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    assert (o_buf[B * H * N * d:] == 7.0).all()
    assert (l_buf[B * H * N:] == 7.0).all()


def test_runs_on_a_side_stream():
    B, H, N, d = 1, 4, 256, 64
    q, k, v = fwd_inputs(B, H, N, d, 31, device="cuda")
    s = torch.cuda.Stream()
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        ea.attn_fwd(q, k, v, o, lse, False, 0.125, stream=s)
    s.synchronize()
    O_ref, L_ref = oracle_fwd(q, k, v, 0.125, False)
    assert_within(compare_fwd(o, lse, O_ref, L_ref, range(B * H), None))


@pytest.mark.parametrize("d", [64, 128])
def test_concurrent_launches_on_several_streams(d):
    """The persistent forward hands out work items from a counter that each
    launch takes for itself: launches running at the same time on different
    streams (and more launches than there are counters) each compute their own
    result, equal to the same call made alone."""
    B, H, N = 2, 8, 1024
    streams = [torch.cuda.Stream() for _ in range(4)]
    ins = [fwd_inputs(B, H, N, d, 40 + n, device="cuda") for n in range(4)]
    refs = []
    for q, k, v in ins:
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        ea.attn_fwd(q, k, v, o, lse, True, d ** -0.5)
        refs.append((o, lse))
    torch.cuda.synchronize()
    outs = [(torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device="cuda"))
            for q, _, _ in ins]
    for rep in range(80):   # 320 launches in flight in groups of four
        for s, (q, k, v), (o, lse) in zip(streams, ins, outs):
            with torch.cuda.stream(s):
                ea.attn_fwd(q, k, v, o, lse, True, d ** -0.5, stream=s)
    torch.cuda.synchronize()
    for (o, lse), (o_ref, l_ref) in zip(outs, refs):
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert ea.attn_get_device_status() == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_partial_items_among_full_items(d, causal):
    """N = 640 leaves each head one work item whose last query tile lies past
    N (at d = 64 an item is three 128-row tiles, at d = 128 two) next to full
    items, and 256 heads give every persistent CTA several of both kinds in
    turn, so the per-buffer barrier phases must stay in step across items
    that skip a tile."""
    B, H, N = 4, 64, 640
    q, k, v = fwd_inputs(B, H, N, d, 71 + d + causal, device="cuda")
    scale = d ** -0.5
    o, lse = _run(q, k, v, causal, scale)
    assert ea.attn_get_device_status() == 0
    heads = [0, 1, 2, 75, 151, 152, 153, 200, 254, 255]
    O_ref, L_ref = oracle_fwd(q, k, v, scale, causal, heads=heads)
    assert_within(compare_fwd(o, lse, O_ref, L_ref, heads, None))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_many_short_items_per_persistent_cta(d, causal):
    """A grid of one CTA per SM over far more (head, query block) items than
    SMs, each only one or two K/V tiles long: every CTA runs a long sequence
    of items, so item hand-over, the per-item barrier phases and the reuse of
    Q, staging and accumulators across items are all exercised.  Heads at the
    start, middle and end of the item order are checked in full."""
    B, H, N = 24, 32, 200                # 768 heads, 768 items
    q, k, v = fwd_inputs(B, H, N, d, 61 + d + causal, device="cuda")
    scale = d ** -0.5
    o, lse = _run(q, k, v, causal, scale)
    heads = [0, 1, 151, 152, 383, 384, 700, B * H - 1]
    O_ref, L_ref = oracle_fwd(q, k, v, scale, causal, heads=heads)
    assert_within(compare_fwd(o, lse, O_ref, L_ref, heads, None))
