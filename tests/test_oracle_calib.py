"""Pins for the oracle's calibration reduction (§3.1, Eq. (1), App. B.1)."""

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(5)


def _random_causal_rows(N, T):
    A = RNG.random((N, T, T)) ** 3
    A = np.tril(A)
    return A / A.sum(axis=2, keepdims=True)


def test_golden_svar(golden):
    g = golden("calib_svar_N2_T2.txt")
    A = np.stack([g["A0"], g["A1"]])
    np.testing.assert_allclose(oracle.calib_mean(A), g["Ahat"], atol=1e-15)
    assert abs(oracle.calib_svar(A) - g["s_var"][0]) < 1e-16


def test_identical_samples_have_zero_variance():
    A = np.repeat(_random_causal_rows(1, 12), 9, axis=0)
    assert oracle.calib_svar(A) < 1e-30   # zero up to the rounding of sum/N


def test_two_sample_closed_form():
    A = _random_causal_rows(2, 15)
    want = ((A[0] - A[1]) ** 2).sum() / (2 * 15 * 15)
    assert abs(oracle.calib_svar(A) - want) < 1e-15


def test_mean_rows_are_causal_distributions():
    Ahat = oracle.calib_mean(_random_causal_rows(7, 20))
    np.testing.assert_allclose(Ahat.sum(1), 1.0, atol=1e-13)
    assert np.all(Ahat[np.triu_indices(20, 1)] == 0)


def test_permutation_invariance():
    A = _random_causal_rows(11, 9)
    s = oracle.calib_svar(A)
    assert abs(oracle.calib_svar(A[RNG.permutation(11)]) - s) < 1e-15


def test_mean_optimality_decomposition():
    # App. B.1: R(P) = R(E[A]) + ||P - E[A]||_F^2 / T^2, and the minimum risk
    # is the (biased) variance: s_var = N / (N - 1) R(A_hat).
    N, T = 13, 10
    A = _random_causal_rows(N, T)
    Ahat = oracle.calib_mean(A)
    for _ in range(5):
        P = _random_causal_rows(1, T)[0]
        lhs = oracle.reconstruction_risk(P, A)
        rhs = oracle.reconstruction_risk(Ahat, A) + ((P - Ahat) ** 2).sum() / T ** 2
        assert abs(lhs - rhs) < 1e-12
    assert abs(oracle.calib_svar(A) - N / (N - 1) * oracle.reconstruction_risk(Ahat, A)) < 1e-15


def test_mean_svar_over_heads_matches_per_head():
    N, nh, T = 4, 3, 6
    A_all = np.stack([_random_causal_rows(N, T) for _ in range(nh)], axis=1)
    Ahat, s = oracle.calib_mean_svar(A_all)
    for h in range(nh):
        np.testing.assert_array_equal(Ahat[h], oracle.calib_mean(A_all[:, h]))
        assert s[h] == oracle.calib_svar(A_all[:, h])


def test_num_select_rounds_half_to_even():
    assert oracle.num_select(0.25, 144) == 36
    assert oracle.num_select(0.125, 12) == 2      # 1.5 -> 2
    assert oracle.num_select(0.25, 10) == 2       # 2.5 -> 2
    assert oracle.num_select(0.5, 12) == 6
    assert oracle.num_select(0.0, 12) == 0
    assert oracle.num_select(1.0, 12) == 12


def test_selection_matches_brute_force_with_index_tiebreak():
    s = RNG.integers(0, 5, size=40).astype(float) / 7.0  # many ties
    for k in (0, 1, 9, 40):
        got = oracle.select_heads(s, k)
        left = list(range(40))
        want = []
        for _ in range(k):
            best = left[0]
            for i in left[1:]:
                if s[i] < s[best]:
                    best = i
            want.append(best)
            left.remove(best)
        assert list(got) == want


def test_kl_score_closed_forms():
    # identical samples: every row KL is zero
    A = np.repeat(_random_causal_rows(1, 10), 5, axis=0)
    assert abs(oracle.calib_kl_score(A)) < 1e-14
    # two samples whose rows are point masses at different keys: for the row
    # i >= 1 with masses on j0 != j1, A_hat = (1/2, 1/2) there and each sample's
    # KL is log 2; row 0 has a single key and contributes nothing
    T = 6
    A = np.zeros((2, T, T))
    for i in range(T):
        A[0, i, 0] = 1.0
        A[1, i, i] = 1.0
    want = (T - 1) * 2 * np.log(2.0) / (2 * T)
    assert abs(oracle.calib_kl_score(A) - want) < 1e-14


def test_kl_score_is_nonnegative_and_permutation_invariant():
    A = _random_causal_rows(9, 12)
    s = oracle.calib_kl_score(A)
    assert s > 0
    assert abs(oracle.calib_kl_score(A[RNG.permutation(9)]) - s) < 1e-14


def test_sharp_mean_reduces_to_the_library_softmax_for_one_sample():
    # N = 1: the mean of the logits is the logits; compare with torch's softmax
    import torch
    T = 9
    L = RNG.normal(size=(1, T, T)) * 3.0
    mask = np.tril(np.ones((T, T), dtype=bool))
    ref = torch.softmax(torch.from_numpy(np.where(mask, L[0], -np.inf)), dim=-1).numpy()
    np.testing.assert_allclose(oracle.sharp_mean_pattern(L), ref, rtol=1e-13, atol=1e-15)


def test_sharp_mean_closed_form_and_jensen_gap():
    # T = 2, row 1: logits (0, 0) and (2, 0) average to (1, 0), so the pattern
    # row is (e, 1) / (e + 1); the post-softmax mean of the same two rows is
    # ((1/2 + e^2/(e^2 + 1)) / 2, ...), which differs.
    L = np.zeros((2, 2, 2))
    L[1, 1, 0] = 2.0
    P = oracle.sharp_mean_pattern(L)
    e = np.e
    np.testing.assert_allclose(P, [[1.0, 0.0], [e / (e + 1), 1 / (e + 1)]], rtol=1e-14)
    soft = 0.5 * (0.5 + e * e / (e * e + 1))
    assert abs(P[1, 0] - soft) > 1e-3


def test_sharp_mean_rows_are_causal_distributions_and_shift_invariant():
    T = 11
    L = RNG.normal(size=(4, T, T))
    P = oracle.sharp_mean_pattern(L)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=1e-13)
    assert np.all(np.triu(P, 1) == 0)
    # adding a per-(sample, row) constant to the logits changes nothing
    shift = RNG.normal(size=(4, T, 1))
    np.testing.assert_allclose(oracle.sharp_mean_pattern(L + shift), P, rtol=1e-12, atol=1e-15)
