"""Pins for the oracle's frozen-head pattern (Eq. (3)) and its forward.

Each test fixes the oracle to something other than itself: a hand-worked
fixture, a closed form, an invariant, or the oracle's own dynamic path under
a construction that must reproduce the same distribution.
"""

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(1234)


def test_golden_pattern_and_output(golden):
    g = golden("static_pattern_T4.txt")
    P = oracle.static_pattern(g["alpha"], g["rho"])
    np.testing.assert_allclose(P, g["P"], rtol=0, atol=1e-15)
    out, logZ = oracle.static_head_fwd(g["alpha"], g["rho"], g["V"])
    np.testing.assert_allclose(out, g["O"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(logZ, g["logZ"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(logZ, oracle.static_log_normaliser(g["alpha"], g["rho"]))


@pytest.mark.parametrize("T", [1, 7, 64])
def test_rows_are_causal_distributions(T):
    alpha = RNG.normal(size=T)
    rho = -np.log1p(np.arange(T)) + RNG.normal(0, 0.3, size=T)
    P = oracle.static_pattern(alpha, rho)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert np.all(P[np.triu_indices(T, 1)] == 0.0)
    assert np.all(P[np.tril_indices(T)] > 0.0)


def test_zero_parameters_give_causal_running_mean():
    T, d = 33, 5
    V = RNG.normal(size=(T, d))
    out, logZ = oracle.static_head_fwd(np.zeros(T), np.zeros(T), V)
    expect = np.cumsum(V, axis=0) / np.arange(1, T + 1)[:, None]
    np.testing.assert_allclose(out, expect, rtol=0, atol=1e-13)
    np.testing.assert_allclose(logZ, np.log(np.arange(1, T + 1)), atol=1e-13)


def test_distance_zero_only_gives_identity():
    T, d = 20, 3
    V = RNG.normal(size=(T, d))
    rho = np.full(T, -np.inf)
    rho[0] = 0.0
    out, _ = oracle.static_head_fwd(RNG.normal(size=T), rho, V)
    np.testing.assert_allclose(out, V, rtol=0, atol=1e-14)


def test_shift_invariance():
    T = 40
    alpha = RNG.normal(size=T)
    rho = RNG.normal(size=T)
    P = oracle.static_pattern(alpha, rho)
    np.testing.assert_allclose(oracle.static_pattern(alpha + 3.7, rho), P, atol=1e-14)
    np.testing.assert_allclose(oracle.static_pattern(alpha, rho - 11.0), P, atol=1e-14)


def test_geometric_closed_form():
    # alpha = 0, rho(d) = -lam d: row i weights q^(i-j) / sum_{m=0..i} q^m.
    T, lam = 25, 0.4
    q = np.exp(-lam)
    P = oracle.static_pattern(np.zeros(T), -lam * np.arange(T))
    for i in range(T):
        norm = (1 - q ** (i + 1)) / (1 - q)
        for j in range(T):
            want = q ** (i - j) / norm if j <= i else 0.0
            assert abs(P[i, j] - want) < 1e-14


def test_cross_path_static_equals_rank1_dynamic():
    # With rho(d) = -lam d, alpha(j) + rho(i-j) = (alpha(j) + lam j) - lam i;
    # the -lam i term is constant along a row, so P equals the causal softmax
    # of the rank-1 scores q_i k_j / sqrt(d) with q_i = (sqrt(d), 0, ...) and
    # k_j = (alpha(j) + lam j, 0, ...).
    T, d, lam = 48, 8, 0.15
    alpha = RNG.normal(size=T)
    rho = -lam * np.arange(T)
    q = np.zeros((T, d)); q[:, 0] = np.sqrt(d)
    k = np.zeros((T, d)); k[:, 0] = alpha + lam * np.arange(T)
    v = RNG.normal(size=(T, d))
    out_dyn, _, A = oracle.dynamic_head_fwd(q, k, v)
    P = oracle.static_pattern(alpha, rho)
    np.testing.assert_allclose(P, A, rtol=0, atol=1e-13)
    out_st, _ = oracle.static_head_fwd(alpha, rho, v)
    np.testing.assert_allclose(out_st, out_dyn, rtol=0, atol=1e-12)


def test_hybrid_routes_heads_and_batches():
    B, H, T, d = 2, 3, 16, 4
    Q, K, V = (RNG.normal(size=(B, H, T, d)) for _ in range(3))
    alpha, rho = RNG.normal(size=(H, T)), RNG.normal(size=(H, T))
    mask = np.array([0, 1, 0], dtype=np.uint8)
    out, lse = oracle.hybrid_attn_fwd(Q, K, V, alpha, rho, mask)
    for b in range(B):
        o, l, _ = oracle.dynamic_head_fwd(Q[b, 0], K[b, 0], V[b, 0])
        np.testing.assert_array_equal(out[b, 0], o)
        np.testing.assert_array_equal(lse[b, 0], l)
        o, l = oracle.static_head_fwd(alpha[1], rho[1], V[b, 1])
        np.testing.assert_array_equal(out[b, 1], o)
        np.testing.assert_array_equal(lse[b, 1], l)
    # static heads never read Q/K
    Q2 = Q.copy(); Q2[:, 1] = np.nan
    out2, _ = oracle.hybrid_attn_fwd(Q2, K, V, alpha, rho, mask)
    np.testing.assert_array_equal(out2, out)


def test_row_restricted_forms_match_full():
    T, d = 50, 4
    q, k, v = (RNG.normal(size=(T, d)) for _ in range(3))
    alpha, rho = RNG.normal(size=T), RNG.normal(size=T)
    rows = [0, 1, 17, 49]
    o, l, _ = oracle.dynamic_head_fwd(q, k, v)
    orow, lrow = oracle.dynamic_head_fwd_rows(q, k, v, rows)
    np.testing.assert_allclose(orow, o[rows], atol=1e-14)
    np.testing.assert_allclose(lrow, l[rows], atol=1e-14)
    o, l = oracle.static_head_fwd(alpha, rho, v)
    orow, lrow = oracle.static_head_fwd_rows(alpha, rho, v, rows)
    np.testing.assert_allclose(orow, o[rows], atol=1e-14)
    np.testing.assert_allclose(lrow, l[rows], atol=1e-14)
