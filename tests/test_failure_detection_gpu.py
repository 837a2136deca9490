"""Failure detection on the GPU, without faulting or hanging it.

Every mbarrier wait in the kernels is bounded.  The self-test entry point makes
one warp wait, through the same bounded-wait routine, on a barrier phase that
nothing completes; the wait must give up after the requested limit, record
ATTN_ERR_TIMEOUT in the device status word, and leave the CUDA context usable
(a forward call afterwards still matches the oracle).
"""
import time

import pytest
import torch

import exact_attention_tma_gb300 as ea
from exact_attention_tma_gb300.inputs import fwd_inputs
from parity import assert_within, compare_fwd, oracle_fwd

pytestmark = pytest.mark.gpu

OK, TIMEOUT = 0, 7


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_ok):
    from exact_attention_tma_gb300 import build

    build.build()
    ea.load()
    assert ea.attn_get_device_status() == OK   # start from a clean status word


def test_expired_wait_reports_timeout_and_context_survives():
    t0 = time.perf_counter()
    ea.attn_selftest_bounded_wait(50)
    status = ea.attn_get_device_status()       # synchronises the stream
    elapsed = time.perf_counter() - t0
    assert status == TIMEOUT
    assert 0.04 <= elapsed < 5.0, elapsed      # gave up after ~50 ms, did not hang
    assert ea.attn_get_device_status() == OK   # reading cleared it
    # The context is still usable: a forward call right after is correct.
    q, k, v = fwd_inputs(1, 2, 300, 64, 5, device="cuda")
    o, lse = ea.forward(q, k, v, causal=True, scale=0.125)
    torch.cuda.synchronize()
    O_ref, L_ref = oracle_fwd(q, k, v, 0.125, True)
    assert_within(compare_fwd(o, lse, O_ref, L_ref, range(2), None))
    assert ea.attn_get_device_status() == OK
