"""Pins for the oracle's attention backward (CPU only).

The pages print no gradient formula ("Why Fast GPUs Still Wait for Memory",
"FlashAttention is an IO algorithm", only says the backward pass recomputes
S), so the oracle's chain rule is pinned here by things other than itself:
central finite differences of the (separately pinned) forward, closed forms
for uniform attention and constant values, a one-key head, and torch's
autograd of the plain softmax-attention expression in float64.
"""
import numpy as np
import pytest
import torch

import oracle


def _loss(Q, K, V, dO, scale, causal):
    O, _ = oracle.attention_head(Q, K, V, scale, causal)
    return float(np.sum(O * dO))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d", [(1, 2), (4, 3), (6, 2)])
def test_gradients_match_central_differences_of_the_forward(n, d, causal):
    rng = np.random.default_rng(n * 10 + d + causal)
    Q, K, V, dO = (rng.standard_normal((n, d)) for _ in range(4))
    scale = 0.8
    dQ, dK, dV = oracle.attention_backward_head(Q, K, V, dO, scale, causal)
    h = 1e-6
    for X, G in ((Q, dQ), (K, dK), (V, dV)):
        for idx in np.ndindex(X.shape):
            keep = X[idx]
            X[idx] = keep + h
            up = _loss(Q, K, V, dO, scale, causal)
            X[idx] = keep - h
            dn = _loss(Q, K, V, dO, scale, causal)
            X[idx] = keep
            assert abs((up - dn) / (2 * h) - G[idx]) < 1e-7, (idx, G[idx], (up - dn) / (2 * h))


def test_uniform_attention_spreads_do_evenly_over_values():
    # Identical keys (non-causal): P = 1/n everywhere, so dV_j = mean_i dO_i
    # for every j, and dS = P (dP - rowmean(dP)).
    rng = np.random.default_rng(3)
    n, d = 7, 4
    Q = rng.standard_normal((n, d))
    K = np.tile(rng.standard_normal((1, d)), (n, 1))
    V, dO = rng.standard_normal((n, d)), rng.standard_normal((n, d))
    dQ, dK, dV = oracle.attention_backward_head(Q, K, V, dO, 0.5, False)
    assert np.allclose(dV, np.tile(dO.mean(0), (n, 1)), atol=1e-14)
    # With equal keys, dQ = scale * sum_j dS_ij k = 0 because rows of dS sum to 0.
    assert np.abs(dQ).max() < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_constant_values_give_zero_query_and_key_gradients(causal):
    # O = v for every row whatever P is, so O does not depend on Q or K.
    rng = np.random.default_rng(4)
    n, d = 6, 3
    Q, K, dO = (rng.standard_normal((n, d)) for _ in range(3))
    V = np.tile(rng.standard_normal((1, d)), (n, 1))
    dQ, dK, dV = oracle.attention_backward_head(Q, K, V, dO, 1.1, causal)
    assert np.abs(dQ).max() < 1e-13 and np.abs(dK).max() < 1e-13
    # dV still routes dO through P: its rows sum over j to sum_i dO_i.
    assert np.allclose(dV.sum(0), dO.sum(0), atol=1e-13)


def test_causal_last_key_is_seen_only_by_the_last_query():
    # Key n-1 is visible to query n-1 alone, so dV_{n-1} = P[n-1, n-1] dO_{n-1};
    # key 0 is the only key of query 0, so P[0, 0] = 1 and dS[0, :] = 0.
    rng = np.random.default_rng(5)
    n, d = 5, 3
    Q, K, V, dO = (rng.standard_normal((n, d)) for _ in range(4))
    _, _, P, _ = oracle.attention_head(Q, K, V, 0.9, True, return_p=True)
    dQ, dK, dV = oracle.attention_backward_head(Q, K, V, dO, 0.9, True)
    assert np.allclose(dV[n - 1], P[n - 1, n - 1] * dO[n - 1], atol=1e-14)
    assert np.abs(dQ[0]).max() < 1e-14


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,H_kv", [(2, 2), (4, 2), (3, 1)])
def test_matches_torch_autograd_in_float64(H, H_kv, causal):
    rng = np.random.default_rng(H * 7 + H_kv + causal)
    B, n, d = 2, 9, 5
    Q = rng.standard_normal((B, H, n, d))
    K = rng.standard_normal((B, H_kv, n, d))
    V = rng.standard_normal((B, H_kv, n, d))
    dO = rng.standard_normal((B, H, n, d))
    scale = 0.37
    dQ, dK, dV = oracle.attention_backward(Q, K, V, dO, scale, causal)

    tq, tk, tv = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (Q, K, V))
    g = H // H_kv
    ke = tk.repeat_interleave(g, dim=1)
    ve = tv.repeat_interleave(g, dim=1)
    s = scale * tq @ ke.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(n, n, dtype=torch.bool).triu(1), float("-inf"))
    o = torch.softmax(s, dim=-1) @ ve
    o.backward(torch.tensor(dO))
    assert np.allclose(dQ, tq.grad.numpy(), atol=1e-12)
    assert np.allclose(dK, tk.grad.numpy(), atol=1e-12)
    assert np.allclose(dV, tv.grad.numpy(), atol=1e-12)


def test_head_subset_returns_unsummed_per_query_head_gradients():
    rng = np.random.default_rng(8)
    Q, dO = rng.standard_normal((1, 4, 6, 2)), rng.standard_normal((1, 4, 6, 2))
    K, V = rng.standard_normal((1, 2, 6, 2)), rng.standard_normal((1, 2, 6, 2))
    dQ, dK, dV = oracle.attention_backward(Q, K, V, dO, 0.5, True)
    sq, sk, sv = oracle.attention_backward(Q, K, V, dO, 0.5, True, heads=[2, 3])
    assert np.array_equal(sq, dQ[0, 2:4])
    assert np.allclose(sk[0] + sk[1], dK[0, 1], atol=1e-15)
    assert np.allclose(sv[0] + sv[1], dV[0, 1], atol=1e-15)
