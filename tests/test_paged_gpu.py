"""GPU parity of the paged-cache decode (attn_decode_paged) against the fp64
oracle's paged decode ("M4.2 GPU Execution Model for Transformer Kernels":
logical K/V continuity does not imply contiguous physical addresses), plus its
device-side bounds check on page ids.
"""
import numpy as np
import pytest
import torch

import exact_attention_tma_gb300 as ea
import oracle
from exact_attention_tma_gb300.inputs import WORKLOADS, paged_decode_inputs, workload_inputs
from parity import O_MAX, O_MEAN, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from exact_attention_tma_gb300 import build

    build.build()
    ea.load()
    yield
    assert ea.attn_get_device_status() == 0


def _run(q, Kp, Vp, table, lens, scale):
    o = torch.empty_like(q)
    ea.attn_decode_paged(q, Kp, Vp, table, lens, o, scale)
    torch.cuda.synchronize()
    return o


def _assert_close(o, O_ref):
    err = np.abs(to_f64(o) - O_ref)
    assert np.isfinite(err).all()
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(4, 4), (8, 2), (8, 1)])
@pytest.mark.parametrize("page_size", [1, 16, 32, 64, 256])
def test_paged_small_full(page_size, H, H_kv, d):
    B, L = 3, 700
    lens = [700, 1, 333]
    q, Kp, Vp, table, sl = paged_decode_inputs(B, H, L, d, page_size, seed=page_size + H + d,
                                               device="cuda", H_kv=H_kv, seq_lens=lens,
                                               extra_pages=5)
    o = _run(q, Kp, Vp, table, sl, d ** -0.5)
    O_ref, _ = oracle.decode_paged(to_f64(q), to_f64(Kp), to_f64(Vp), table.cpu().numpy(),
                                   np.array(lens), d ** -0.5)
    _assert_close(o, O_ref)


def test_paged_equals_contiguous_decode_of_the_same_tokens():
    # The same tokens laid out contiguously through attn_decode_gqa.
    B, H, H_kv, L, d, S = 2, 8, 2, 1000, 128, 32
    q, Kp, Vp, table, sl = paged_decode_inputs(B, H, L, d, S, seed=9, device="cuda", H_kv=H_kv)
    nblk = table.shape[1]
    K = Kp[table.long()].permute(0, 2, 1, 3, 4).reshape(B, H_kv, nblk * S, d)[:, :, :L].contiguous()
    V = Vp[table.long()].permute(0, 2, 1, 3, 4).reshape(B, H_kv, nblk * S, d)[:, :, :L].contiguous()
    o1 = _run(q, Kp, Vp, table, sl, 0.09)
    o2 = torch.empty_like(q)
    ea.attn_decode_gqa(q, K, V, o2, 0.09)
    torch.cuda.synchronize()
    O_ref, _ = oracle.decode_gqa(to_f64(q), to_f64(K), to_f64(V), 0.09)
    _assert_close(o1, O_ref)
    _assert_close(o2, O_ref)


def test_empty_sequence_gives_zero_output():
    q, Kp, Vp, table, sl = paged_decode_inputs(2, 4, 64, 64, 16, seed=4, device="cuda",
                                               seq_lens=[0, 64])
    o = _run(q, Kp, Vp, table, sl, 0.125)
    assert torch.count_nonzero(o[0]) == 0
    O_ref, _ = oracle.decode_paged(to_f64(q[1:]), to_f64(Kp), to_f64(Vp), table[1:].cpu().numpy(),
                                   np.array([64]), 0.125)
    _assert_close(o[1:], O_ref)


def test_bad_page_id_is_reported_not_dereferenced():
    q, Kp, Vp, table, sl = paged_decode_inputs(2, 4, 256, 64, 16, seed=5, device="cuda")
    table[1, 3] = Kp.shape[0] + 1000          # past the pool
    table[0, 0] = -7
    o = torch.empty_like(q)
    ea.attn_decode_paged(q, Kp, Vp, table, sl, o, 0.125)
    assert ea.attn_get_device_status() == ea.ATTN_ERR_ARG
    # the context is still usable and the status word is clear again
    table[1, 3] = 0
    table[0, 0] = 1
    ea.attn_decode_paged(q, Kp, Vp, table, sl, o, 0.125)
    assert ea.attn_get_device_status() == 0


@pytest.mark.parametrize("page_size", [16, 64])
def test_grouped_bad_page_is_skipped_and_reported(page_size):
    # Grouped heads take the tensor-core path: a bad id in sequence 0's first
    # block drops that block's tokens there, sequence 1 is untouched, and the
    # call reports ATTN_ERR_ARG.
    B, H, H_kv, L, d = 2, 8, 2, 300, 128
    q, Kp, Vp, table, sl = paged_decode_inputs(B, H, L, d, page_size, seed=13, device="cuda",
                                               H_kv=H_kv)
    tab = table.cpu().numpy().copy()
    table[0, 0] = -3
    o = torch.empty_like(q)
    ea.attn_decode_paged(q, Kp, Vp, table, sl, o, 0.1)
    assert ea.attn_get_device_status() == ea.ATTN_ERR_ARG
    O1, _ = oracle.decode_paged(to_f64(q[1:]), to_f64(Kp), to_f64(Vp), tab[1:], np.array([L]), 0.1)
    _assert_close(o[1:], O1)
    rows = np.concatenate([np.arange(page_size * blk, min(L, page_size * (blk + 1)))
                           for blk in range(1, tab.shape[1])])
    K0 = np.stack([oracle.paged_rows(to_f64(Kp), tab[0], L, kh)[rows] for kh in range(H_kv)])
    V0 = np.stack([oracle.paged_rows(to_f64(Vp), tab[0], L, kh)[rows] for kh in range(H_kv)])
    O0, _ = oracle.decode_gqa(to_f64(q[:1]), K0[None], V0[None], 0.1)
    _assert_close(o[:1], O0)


def test_paged_gqa_workload_sampled():
    w = WORKLOADS["paged_gqa_decode"]
    q, Kp, Vp, table, sl = workload_inputs(w, device="cuda")
    o = _run(q, Kp, Vp, table, sl, w.scale)
    tab = table.cpu().numpy()
    for flat in [0, 7, 8, 63, 64 * 5 + 33, w.B * w.H - 1]:
        b, h = divmod(flat, w.H)
        kh = oracle.kv_head_of(h, w.H, w.H_kv)
        O_ref, _ = oracle.decode_paged(to_f64(q[b:b + 1, h:h + 1]), to_f64(Kp[:, kh:kh + 1]),
                                       to_f64(Vp[:, kh:kh + 1]), tab[b:b + 1],
                                       np.array([int(sl[b])]), w.scale)
        _assert_close(o[b:b + 1, h:h + 1], O_ref)


def test_paged_workload_sampled():
    w = WORKLOADS["paged_decode"]
    q, Kp, Vp, table, sl = workload_inputs(w, device="cuda")
    o = _run(q, Kp, Vp, table, sl, w.scale)
    tab = table.cpu().numpy()
    for flat in [0, 1, 31, 32, 200, w.B * w.H - 1]:
        b, h = divmod(flat, w.H)
        kh = oracle.kv_head_of(h, w.H, w.H_kv)
        O_ref, _ = oracle.decode_paged(to_f64(q[b:b + 1, h:h + 1]), to_f64(Kp[:, kh:kh + 1]),
                                       to_f64(Vp[:, kh:kh + 1]), tab[b:b + 1],
                                       np.array([int(sl[b])]), w.scale)
        _assert_close(o[b:b + 1, h:h + 1], O_ref)
