"""Pins for the oracle's compact pattern fit (Eq. (3)/(4), App. A.2)."""

import numpy as np

import oracle

RNG = np.random.default_rng(17)


def _random_causal_rows(T):
    A = np.tril(RNG.random((T, T)) ** 2)
    return A / A.sum(axis=1, keepdims=True)


def test_gradient_matches_finite_differences():
    T = 9
    A = _random_causal_rows(T)
    alpha, rho = RNG.normal(size=T), RNG.normal(size=T)
    ga, gr = oracle.fit_gradient(alpha, rho, oracle.marginals(A))
    h = 1e-6
    for vec, g in ((alpha, ga), (rho, gr)):
        for j in range(T):
            old = vec[j]
            vec[j] = old + h
            fp = oracle.fit_loss(alpha, rho, A)
            vec[j] = old - h
            fm = oracle.fit_loss(alpha, rho, A)
            vec[j] = old
            assert abs((fp - fm) / (2 * h) - g[j]) < 1e-8


def test_marginals_are_sufficient_statistics():
    # Two targets with the same column and diagonal sums give the same
    # gradient everywhere (and losses that differ by a constant).
    T = 6
    A = _random_causal_rows(T)
    B = A.copy()
    # a 3x3 move with zero row, column and diagonal sums:
    #   [[t, -t, 0], [-t, 0, t], [0, t, -t]] at rows 3..5, columns 0..2
    t = 0.01
    B[3:6, 0:3] += t * np.array([[1, -1, 0], [-1, 0, 1], [0, 1, -1]])
    np.testing.assert_allclose(B.sum(axis=1), 1.0, atol=1e-15)
    ca, da = oracle.marginals(A)
    cb, db = oracle.marginals(B)
    np.testing.assert_allclose(ca, cb, atol=1e-15)
    np.testing.assert_allclose(da, db, atol=1e-15)
    alpha, rho = RNG.normal(size=T), RNG.normal(size=T)
    ga, gr = oracle.fit_gradient(alpha, rho, (ca, da))
    gb, grb = oracle.fit_gradient(alpha, rho, (cb, db))
    np.testing.assert_allclose(ga, gb, rtol=0, atol=1e-15)
    np.testing.assert_allclose(gr, grb, rtol=0, atol=1e-15)


def test_representable_target_is_recovered():
    T = 24
    alpha_t = 0.5 * RNG.normal(size=T)
    rho_t = -0.3 * np.arange(T) + 0.2 * RNG.normal(size=T)
    A = oracle.static_pattern(alpha_t, rho_t)
    alpha, rho, kl = oracle.compact_fit(A, steps=400)
    kl0 = oracle.mean_row_kl(A, oracle.static_pattern(np.zeros(T), np.zeros(T)))
    assert kl < 2e-3 < kl0
    assert kl == oracle.mean_row_kl(A, oracle.static_pattern(alpha, rho))


def test_kl_is_zero_only_for_equal_rows():
    T = 7
    A = _random_causal_rows(T)
    assert abs(oracle.mean_row_kl(A, A)) < 1e-15
    assert oracle.mean_row_kl(A, oracle.static_pattern(np.zeros(T), np.zeros(T))) > 0


def test_select_fitted_skips_heads_over_the_gate():
    order = [5, 2, 9, 1, 7]
    kls = [0.05, 0.31, 0.2, 0.19, 0.01]
    assert list(oracle.select_fitted(order, kls, 3)) == [5, 9, 1]
    assert list(oracle.select_fitted(order, kls, 10)) == [5, 9, 1, 7]
    assert list(oracle.select_fitted(order, kls, 0)) == []


def test_mean_row_kl_golden(golden):
    # Hand-worked T = 3 case: the direction KL(A_hat || P_hat) and the 1/T row
    # average are both visible in the value.
    g = golden("fit_row_kl_T3.txt")
    want = float(np.sum(g["kl_terms"]))
    assert abs(oracle.mean_row_kl(g["A"], g["P"]) - want) < 1e-14
    # the other direction is a different number (1/4 ln(3/2))
    assert abs(oracle.mean_row_kl(g["P"], g["A"]) - 0.25 * np.log(1.5)) < 1e-14


def test_mean_row_kl_is_cross_entropy_minus_entropy():
    # The gate and the fitted objective are tied: for any causal target A and
    # any (alpha, rho), mean row KL(A || P_hat) = fit_loss - (row entropy of A) / T.
    T = 11
    A = _random_causal_rows(T)
    alpha, rho = RNG.normal(size=T), RNG.normal(size=T)
    m = A > 0
    entropy = -(A[m] * np.log(A[m])).sum()
    kl = oracle.mean_row_kl(A, oracle.static_pattern(alpha, rho))
    assert abs(kl - (oracle.fit_loss(alpha, rho, A) - entropy / T)) < 1e-12


def test_adam_two_steps_golden(golden):
    g = golden("adam_two_steps.txt")
    lr, b1, b2, eps = (float(g[k][0]) for k in ("lr", "b1", "b2", "eps"))
    theta, m, v = np.array([g["theta0"][0]]), np.zeros(1), np.zeros(1)
    for t in (1, 2):
        theta, m, v = oracle.adam_step(theta, np.array([g["g"][t - 1]]), m, v, t, lr, b1, b2, eps)
        assert abs(m[0] - g["m"][t - 1]) < 1e-15
        assert abs(v[0] - g["v"][t - 1]) < 1e-18
        assert abs(theta[0] - g["theta"][t - 1]) < 1e-13
    # a gradient as small as eps: the step is lr / 2 only with eps outside the
    # square root and with the bias correction
    theta, _, _ = oracle.adam_step(np.zeros(1), np.array([g["g_small"][0]]), np.zeros(1),
                                   np.zeros(1), 1, lr, b1, b2, eps)
    assert abs(theta[0] - g["theta_small"][0]) < 1e-12


def test_compact_fit_runs_adam_from_the_log_marginals():
    # One step of compact_fit is one adam_step from the stated initial point.
    T = 7
    A = _random_causal_rows(T)
    col, diag = oracle.marginals(A)
    a0 = np.log(np.maximum(col / (T - np.arange(T)), 1e-30))
    r0 = np.log(np.maximum(diag / (T - np.arange(T)), 1e-30))
    ga, gr = oracle.fit_gradient(a0, r0, (col, diag))
    a1, _, _ = oracle.adam_step(a0, ga, np.zeros(T), np.zeros(T), 1, 1e-2, 0.9, 0.999, 1e-8)
    r1, _, _ = oracle.adam_step(r0, gr, np.zeros(T), np.zeros(T), 1, 1e-2, 0.9, 0.999, 1e-8)
    alpha, rho, kl = oracle.compact_fit(A, steps=1)
    np.testing.assert_allclose(alpha, a1, rtol=0, atol=1e-15)
    np.testing.assert_allclose(rho, r1, rtol=0, atol=1e-15)
