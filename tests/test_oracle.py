"""Pins for the fp64 CPU oracle (no GPU).

The oracle is checked against things fixed by the definition of attention
("Why Fast GPUs Still Wait for Memory", section 'Attention from first
principles': S = QK^T, P = softmax(S), O = PV), not against itself:
hand-worked closed forms (tests/golden/hand_cases.json), invariants that hold
for any input (rows of P sum to one, masked entries are exactly zero,
permutation of keys/values, identical keys, constant V, causal row 0), the
split-KV identity, and brute force in 50-digit arithmetic without the
max-shift on tiny random inputs.  Each pin is chosen so that a plausible slip
in the oracle (dropped scale, transposed operand, wrong mask index, natural
vs base-2 log, missing max add-back, wrong combine weight) fails one of them.
"""
import json
import math
import os

import mpmath
import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")
_NS = {"e": math.e, "ln": math.log, "sqrt": math.sqrt, "inf": math.inf}


def _ev(expr):
    return float(eval(expr, {"__builtins__": {}}, _NS))


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _golden()["cases"], ids=lambda c: c["name"])
def test_hand_cases(case):
    O, LSE = oracle.attention_head(case["Q"], case["K"], case["V"], case["scale"],
                                   case["causal"])
    O_exp = np.array([[_ev(x) for x in row] for row in case["O"]])
    LSE_exp = np.array([_ev(x) for x in case["LSE"]])
    np.testing.assert_allclose(O, O_exp, rtol=0, atol=1e-14)
    np.testing.assert_allclose(LSE, LSE_exp, rtol=0, atol=1e-14)


@pytest.mark.parametrize("case", _golden()["decode_cases"], ids=lambda c: c["name"])
def test_decode_hand_cases(case):
    O, LSE = oracle.decode(case["q"], case["K"], case["V"], case["scale"])
    np.testing.assert_allclose(O, [_ev(x) for x in case["O"]], rtol=0, atol=1e-14)
    assert abs(float(LSE) - _ev(case["LSE"])) < 1e-14
    O_s, lse_s = oracle.decode_split(case["q"], case["K"], case["V"], case["scale"],
                                     case["nsplit"])
    np.testing.assert_allclose(O_s, [[_ev(x) for x in r] for r in case["O_s"]],
                               rtol=0, atol=1e-14)
    for got, want in zip(lse_s, case["lse_s"]):
        w = _ev(want)
        if w == -math.inf:
            assert got == -math.inf
        else:
            assert abs(got - w) < 1e-14
    O_c, LSE_c = oracle.lse_combine(O_s, lse_s)
    np.testing.assert_allclose(O_c, [_ev(x) for x in case["O"]], rtol=0, atol=1e-14)
    assert abs(LSE_c - _ev(case["LSE"])) < 1e-14


def _rand(rng, n, d, std=1.0):
    return rng.standard_normal((n, d)) * std


@pytest.mark.parametrize("causal", [False, True])
def test_rows_of_p_sum_to_one_and_mask_is_exact(causal):
    rng = np.random.default_rng(11)
    N, d = 37, 8
    Q, K, V = _rand(rng, N, d, 2.0), _rand(rng, N, d, 2.0), _rand(rng, N, d)
    O, LSE, P, err = oracle.attention_head(Q, K, V, 0.7, causal, return_p=True)
    assert err < 1e-14
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-14, rtol=0)
    assert (P >= 0).all()
    if causal:
        assert (P[np.triu_indices(N, 1)] == 0.0).all()
        assert (P[np.tril_indices(N)] > 0.0).all()
    else:
        assert (P > 0).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("zero_q", [False, True])
def test_identical_keys_give_mean_of_v(causal, zero_q):
    rng = np.random.default_rng(5)
    N, d, scale = 23, 6, 0.37
    Q = np.zeros((N, d)) if zero_q else _rand(rng, N, d)
    k = rng.standard_normal(d)
    K = np.tile(k, (N, 1))
    V = _rand(rng, N, d)
    O, LSE = oracle.attention_head(Q, K, V, scale, causal)
    for i in range(N):
        n_vis = i + 1 if causal else N
        np.testing.assert_allclose(O[i], V[:n_vis].mean(axis=0), atol=1e-13, rtol=0)
        s = scale * float(Q[i] @ k)
        assert abs(LSE[i] - (s + math.log(n_vis))) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_constant_v_gives_constant_output(causal):
    rng = np.random.default_rng(7)
    N, d = 19, 5
    v = rng.standard_normal(d)
    O, _ = oracle.attention_head(_rand(rng, N, d, 3.0), _rand(rng, N, d, 3.0),
                                 np.tile(v, (N, 1)), 0.5, causal)
    np.testing.assert_allclose(O, np.tile(v, (N, 1)), atol=1e-13, rtol=0)


def test_causal_row0_is_v0():
    rng = np.random.default_rng(9)
    N, d, scale = 16, 4, 0.81
    Q, K, V = _rand(rng, N, d), _rand(rng, N, d), _rand(rng, N, d)
    O, LSE = oracle.attention_head(Q, K, V, scale, True)
    assert (O[0] == V[0]).all()
    assert abs(LSE[0] - scale * float(Q[0] @ K[0])) < 1e-15


def test_permuting_keys_and_values_together_is_invariant():
    rng = np.random.default_rng(13)
    N, d = 29, 7
    Q, K, V = _rand(rng, N, d), _rand(rng, N, d), _rand(rng, N, d)
    perm = rng.permutation(N)
    O1, L1 = oracle.attention_head(Q, K, V, 0.4, False)
    O2, L2 = oracle.attention_head(Q, K[perm], V[perm], 0.4, False)
    np.testing.assert_allclose(O1, O2, atol=1e-13, rtol=0)
    np.testing.assert_allclose(L1, L2, atol=1e-13, rtol=0)


def test_large_scores_stay_finite():
    # Identical keys with huge scores: exp without the shift would overflow.
    N, d = 8, 2
    Q = np.full((N, d), 30.0)
    K = np.full((N, d), 30.0)
    V = np.arange(N * d, dtype=np.float64).reshape(N, d)
    O, LSE = oracle.attention_head(Q, K, V, 1.0, False)
    np.testing.assert_allclose(O, np.tile(V.mean(axis=0), (N, 1)), atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, 1800.0 + math.log(N), atol=1e-12, rtol=0)


def test_row_subset_matches_full():
    rng = np.random.default_rng(17)
    N, d = 41, 9
    Q, K, V = _rand(rng, N, d), _rand(rng, N, d), _rand(rng, N, d)
    for causal in (False, True):
        O, LSE = oracle.attention_head(Q, K, V, 0.3, causal)
        rows = [40, 0, 17, 3]
        Os, Ls = oracle.attention_head(Q, K, V, 0.3, causal, rows=rows)
        np.testing.assert_array_equal(Os, O[rows])
        np.testing.assert_array_equal(Ls, LSE[rows])


@pytest.mark.parametrize("L,nsplit", [(1, 1), (1, 32), (7, 3), (64, 32), (100, 32),
                                      (257, 32), (8192 // 16, 32)])
def test_split_then_combine_equals_unsplit(L, nsplit):
    rng = np.random.default_rng(L * 131 + nsplit)
    d = 16
    q, K, V = rng.standard_normal(d) * 2, _rand(rng, L, d, 2.0), _rand(rng, L, d)
    O, LSE = oracle.decode(q, K, V, 0.25)
    O_s, lse_s = oracle.decode_split(q, K, V, 0.25, nsplit)
    O_c, LSE_c = oracle.lse_combine(O_s, lse_s)
    np.testing.assert_allclose(O_c, O, atol=1e-12, rtol=0)
    assert abs(LSE_c - float(LSE)) < 1e-12
    chunk = -(-L // nsplit)
    for s in range(nsplit):
        if s * chunk >= L:
            assert lse_s[s] == -math.inf and (O_s[s] == 0).all()


def _brute(Q, K, V, scale, causal):
    """Softmax in 50-digit arithmetic with no max shift (independent of the C code)."""
    mpmath.mp.dps = 50
    nq, d = len(Q), len(Q[0])
    nk = len(K)
    O = np.zeros((nq, d))
    LSE = np.zeros(nq)
    for i in range(nq):
        w = []
        for j in range(nk):
            if causal and j > i:
                w.append(mpmath.mpf(0))
                continue
            dot = mpmath.fsum(mpmath.mpf(float(Q[i][k])) * mpmath.mpf(float(K[j][k]))
                              for k in range(d))
            w.append(mpmath.exp(mpmath.mpf(scale) * dot))
        z = mpmath.fsum(w)
        for k in range(d):
            O[i, k] = float(mpmath.fsum(w[j] * mpmath.mpf(float(V[j][k]))
                                        for j in range(nk)) / z)
        LSE[i] = float(mpmath.log(z))
    return O, LSE


@pytest.mark.parametrize("seed", range(6))
def test_bruteforce_tiny_random(seed):
    rng = np.random.default_rng(1000 + seed)
    N = int(rng.integers(1, 9))
    d = int(rng.integers(1, 5))
    scale = float(rng.uniform(0.1, 2.0))
    Q, K, V = _rand(rng, N, d, 1.5), _rand(rng, N, d, 1.5), _rand(rng, N, d)
    for causal in (False, True):
        O, LSE = oracle.attention_head(Q, K, V, scale, causal)
        Ob, Lb = _brute(Q, K, V, scale, causal)
        np.testing.assert_allclose(O, Ob, atol=1e-13, rtol=0)
        np.testing.assert_allclose(LSE, Lb, atol=1e-13, rtol=0)


def test_rectangular_noncausal_bruteforce():
    # Decode is the one-row, non-causal case against a longer key list.
    rng = np.random.default_rng(77)
    L, d = 11, 3
    q, K, V = rng.standard_normal(d), _rand(rng, L, d), _rand(rng, L, d)
    O, LSE = oracle.decode(q, K, V, 0.9)
    Ob, Lb = _brute([q], K, V, 0.9, False)
    np.testing.assert_allclose(O, Ob[0], atol=1e-13, rtol=0)
    assert abs(float(LSE) - Lb[0]) < 1e-13


def test_batched_wrapper_matches_per_head():
    rng = np.random.default_rng(3)
    B, H, N, d = 2, 3, 10, 4
    Q = rng.standard_normal((B, H, N, d))
    K = rng.standard_normal((B, H, N, d))
    V = rng.standard_normal((B, H, N, d))
    O, LSE = oracle.attention(Q, K, V, 0.5, True, threads=3)
    for b in range(B):
        for h in range(H):
            o, l = oracle.attention_head(Q[b, h], K[b, h], V[b, h], 0.5, True)
            np.testing.assert_array_equal(O[b, h], o)
            np.testing.assert_array_equal(LSE[b, h], l)


def test_bad_arguments_are_rejected():
    with pytest.raises(RuntimeError):
        # causal needs as many queries as keys
        oracle.attention_head(np.ones((2, 2)), np.ones((3, 2)), np.ones((3, 2)), 1.0, True)
    with pytest.raises(RuntimeError):
        oracle.attention_head(np.ones((2, 2)), np.ones((2, 2)), np.ones((2, 2)), 1.0,
                              False, rows=[5])


# ---------------------------------------------------------------- grouped heads
# "Why Fast GPUs Still Wait for Memory", section "Attention III · KV cache, GQA,
# MLA": h query heads share h_kv K/V heads, group size g = h / h_kv.  Reading:
# contiguous groups, query head h -> K/V head floor(h / g).

def test_kv_head_mapping_contiguous_groups():
    assert [oracle.kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [oracle.kv_head_of(h, 4, 4) for h in range(4)] == [0, 1, 2, 3]
    assert [oracle.kv_head_of(h, 6, 1) for h in range(6)] == [0] * 6   # MQA
    with pytest.raises(ValueError):
        oracle.kv_head_of(0, 6, 4)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_constant_values_per_kv_head(causal):
    # Each K/V head holds one constant value row, so every query head must
    # return exactly its group's value: a mapping mistake (h % h_kv, say)
    # would hand heads 1 and 2 the wrong constant.
    rng = np.random.default_rng(11)
    B, H, H_kv, N, d = 2, 4, 2, 6, 3
    Q = rng.standard_normal((B, H, N, d))
    K = rng.standard_normal((B, H_kv, N, d))
    vals = np.array([[1.0, -2.0, 0.5], [3.0, 0.25, -1.0]])
    V = np.empty((B, H_kv, N, d))
    for b in range(B):
        for kh in range(H_kv):
            V[b, kh] = vals[kh] + 10.0 * b
    O, LSE = oracle.attention_gqa(Q, K, V, 0.7, causal)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(O[b, h], np.tile(vals[h // 2] + 10.0 * b, (N, 1)),
                                       rtol=0, atol=1e-12)
    q = rng.standard_normal((B, H, d))
    Od, _ = oracle.decode_gqa(q, K, V, 0.7)
    for b in range(B):
        for h in range(H):
            np.testing.assert_allclose(Od[b, h], vals[h // 2] + 10.0 * b, rtol=0, atol=1e-12)


def test_gqa_with_one_group_per_head_is_mha():
    rng = np.random.default_rng(12)
    Q, K, V = (rng.standard_normal((2, 3, 5, 4)) for _ in range(3))
    O, LSE = oracle.attention_gqa(Q, K, V, 0.5, True)
    O2, LSE2 = oracle.attention(Q, K, V, 0.5, True)
    np.testing.assert_array_equal(O, O2)
    np.testing.assert_array_equal(LSE, LSE2)
    q = rng.standard_normal((2, 3, 4))
    Od, Ld = oracle.decode_gqa(q, K, V, 0.5)
    Od2, Ld2 = oracle.decode(q, K, V, 0.5)
    np.testing.assert_array_equal(Od, Od2)
    np.testing.assert_array_equal(Ld, Ld2)


# ---------------------------------------------------------------- paged caches
# "M4.2 - GPU Execution Model for Transformer Kernels": logical K/V continuity
# does not imply contiguous physical addresses.  Reading: block table of page
# ids per sequence, token t in page table[t // page_size], slot t % page_size.

def _scatter_to_pages(K, V, page_size, rng, extra_pages=3):
    """Contiguous (B, H_kv, L, d) caches -> shuffled K/V pages and one block table."""
    B, H_kv, L, d = K.shape
    nblk = -(-L // page_size)
    n_pages = B * nblk + extra_pages
    perm = rng.permutation(n_pages)[: B * nblk].reshape(B, nblk)
    Kp = rng.standard_normal((n_pages, H_kv, page_size, d))   # junk everywhere else
    Vp = rng.standard_normal((n_pages, H_kv, page_size, d))
    for b in range(B):
        for i in range(nblk):
            t0, t1 = i * page_size, min(L, (i + 1) * page_size)
            Kp[perm[b, i], :, : t1 - t0] = K[b, :, t0:t1]
            Vp[perm[b, i], :, : t1 - t0] = V[b, :, t0:t1]
    return Kp, Vp, perm


@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_paged_decode_equals_contiguous_decode(page_size):
    rng = np.random.default_rng(21)
    B, H, H_kv, L, d = 3, 4, 2, 37, 8
    q = rng.standard_normal((B, H, d))
    K = rng.standard_normal((B, H_kv, L, d))
    V = rng.standard_normal((B, H_kv, L, d))
    Kp, Vp, table = _scatter_to_pages(K, V, page_size, rng)
    lens = np.array([L, 1, 20])
    O, LSE = oracle.decode_paged(q, Kp, Vp, table, lens, 0.3)
    for b in range(B):
        Ob, Lb = oracle.decode_gqa(q[b:b + 1], K[b:b + 1, :, : lens[b]], V[b:b + 1, :, : lens[b]], 0.3)
        np.testing.assert_allclose(O[b], Ob[0], rtol=0, atol=1e-13)
        np.testing.assert_allclose(LSE[b], Lb[0], rtol=0, atol=1e-13)


def test_paged_rows_follow_the_block_table():
    # token t -> page table[t // S], slot t % S; a transposed index would fail.
    S = 3
    pages = np.arange(5 * 1 * S * 1, dtype=np.float64).reshape(5, 1, S, 1)
    table = np.array([4, 0, 2])
    rows = oracle.paged_rows(pages, table, 7, 0)[:, 0]
    assert list(rows) == [12, 13, 14, 0, 1, 2, 6]


# ---------------------------------------------------------------- FP8 (E4M3)
def test_e4m3_decoder_matches_torch_for_every_code():
    torch = pytest.importorskip("torch")
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode_e4m3(codes.numpy())
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    keep = ~np.isnan(ref)
    assert np.array_equal(ref[keep], got[keep])


@pytest.mark.parametrize("code,value", [
    (0x00, 0.0), (0x38, 1.0), (0x40, 2.0), (0x3C, 1.5), (0x7E, 448.0), (0xFE, -448.0),
    (0x08, 2.0 ** -6), (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0xB8, -1.0),
])
def test_e4m3_hand_values(code, value):
    # Sign | exponent (bias 7) | 3-bit mantissa; exponent 0 is subnormal.
    assert oracle.e4m3_value(code) == value


def test_e4m3_nan_codes_and_negative_zero():
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))
    z = oracle.e4m3_value(0x80)
    assert z == 0.0 and math.copysign(1.0, z) == -1.0


def test_fp8_attention_is_attention_of_the_descaled_values():
    # Codes 0x38 (1.0) and 0x40 (2.0) with descales: every score equals
    # scale * dq * dk * 1 * 2 * d, so P is uniform and O is the mean of V.
    d, n = 4, 3
    Q8 = np.full((n, d), 0x38, np.uint8)
    K8 = np.full((n, d), 0x40, np.uint8)
    V8 = np.array([[0x38] * d, [0x40] * d, [0x3C] * d], np.uint8)
    O, L = oracle.attention_fp8(Q8[None], K8[None], V8[None], 0.5, 0.25, 2.0, 0.3, False)
    assert np.allclose(O[0], np.full((n, d), 2.0 * (1.0 + 2.0 + 1.5) / 3), atol=1e-15)
    s = 0.3 * 0.5 * 0.25 * 2.0 * d
    assert np.allclose(L[0], s + math.log(n), atol=1e-14)
