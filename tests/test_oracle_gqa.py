"""Pins for the grouped-query form of the oracle: central finite differences
of every gradient on a small case (which checks that a shared K/V head
collects the gradients of all the query heads it serves), the reduction to
the per-head layer when every query head has its own K/V, and the sharing of
K/V inside a group."""

import numpy as np

import oracle

RNG = np.random.default_rng(11)


def _case(B=2, H=4, H_kv=2, T=5, d=3, static=(1, 2)):
    Q = RNG.normal(size=(B, H, T, d))
    K = RNG.normal(size=(B, H_kv, T, d))
    V = RNG.normal(size=(B, H_kv, T, d))
    alpha = RNG.normal(size=(H, T))
    rho = -0.3 * np.arange(T)[None, :] + 0.2 * RNG.normal(size=(H, T))
    mask = np.zeros(H, dtype=bool)
    mask[list(static)] = True
    dO = RNG.normal(size=(B, H, T, d))
    return Q, K, V, alpha, rho, mask, dO


def test_gqa_gradients_match_finite_differences():
    Q, K, V, alpha, rho, mask, dO = _case()

    def loss(Q, K, V, alpha, rho):
        out, _ = oracle.gqa_hybrid_attn_fwd(Q, K, V, alpha, rho, mask)
        return float((out * dO).sum())

    dQ, dK, dV, da, dr = oracle.gqa_hybrid_attn_bwd(Q, K, V, alpha, rho, mask, dO)
    args = [Q, K, V, alpha, rho]
    grads = [dQ, dK, dV, da, dr]
    h = 1e-6
    for ai, (arr, g) in enumerate(zip(args, grads)):
        for idx in [tuple(RNG.integers(0, s) for s in arr.shape) for _ in range(12)]:
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[ai][idx] += h
            minus[ai][idx] -= h
            num = (loss(*plus) - loss(*minus)) / (2 * h)
            assert abs(num - g[idx]) < 1e-6 * max(1.0, abs(num)), (ai, idx, num, g[idx])


def test_gqa_with_one_query_head_per_kv_head_is_the_per_head_layer():
    Q, K, V, alpha, rho, mask, dO = _case(H=3, H_kv=3, static=(1,))
    out, lse = oracle.gqa_hybrid_attn_fwd(Q, K, V, alpha, rho, mask)
    ref_out, ref_lse = oracle.hybrid_attn_fwd(Q, K, V, alpha, rho, mask)
    np.testing.assert_array_equal(out, ref_out)
    np.testing.assert_array_equal(lse, ref_lse)
    got = oracle.gqa_hybrid_attn_bwd(Q, K, V, alpha, rho, mask, dO)
    ref = oracle.hybrid_attn_bwd(Q, K, V, alpha, rho, mask, dO)
    for a, b in zip(got, ref):
        np.testing.assert_array_equal(a, b)


def test_query_heads_of_one_group_share_k_and_v():
    # two dynamic query heads of the same group with equal Q give equal
    # outputs; with the other group's K/V they would not
    Q, K, V, alpha, rho, _, _ = _case(B=1, H=4, H_kv=2, static=())
    mask = np.zeros(4, dtype=bool)
    Q[:, 1] = Q[:, 0]
    Q[:, 2] = Q[:, 0]
    out, _ = oracle.gqa_hybrid_attn_fwd(Q, K, V, alpha, rho, mask)
    np.testing.assert_allclose(out[:, 1], out[:, 0], rtol=1e-15)
    assert np.abs(out[:, 2] - out[:, 0]).max() > 1e-3
