"""Pins for the oracle's backward pass: hand-worked fixtures, central finite
differences in float64, gauge invariance and closed forms."""

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(7)


def test_golden_dynamic_backward(golden):
    g = golden("dynamic_head_T2.txt")
    q, k, v, dO = (g[n][:, None] for n in ("q", "k", "v", "dO"))
    dq, dk, dv = oracle.dynamic_head_bwd(q, k, v, dO)
    np.testing.assert_allclose(dv[:, 0], g["dV"], atol=1e-14)
    np.testing.assert_allclose(dq[:, 0], g["dQ"], atol=1e-14)
    np.testing.assert_allclose(dk[:, 0], g["dK"], atol=1e-14)


def test_golden_static_backward(golden):
    g = golden("static_head_bwd_T2.txt")
    np.testing.assert_allclose(oracle.static_pattern(g["alpha"], g["rho"]), g["P"], atol=1e-15)
    dvs, da, dr = oracle.static_head_bwd(g["alpha"], g["rho"], [g["v"][:, None]], [g["dO"][:, None]])
    np.testing.assert_allclose(dvs[0][:, 0], g["dV"], atol=1e-14)
    np.testing.assert_allclose(da, g["dalpha"], atol=1e-14)
    np.testing.assert_allclose(dr, g["drho"], atol=1e-14)


def _loss(Q, K, V, alpha, rho, mask, dO):
    out, _ = oracle.hybrid_attn_fwd(Q, K, V, alpha, rho, mask)
    return float((out * dO).sum())


def _fd(f, x, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        old = x[idx]
        x[idx] = old + eps
        fp = f()
        x[idx] = old - eps
        fm = f()
        x[idx] = old
        g[idx] = (fp - fm) / (2 * eps)
    return g


def test_finite_differences_all_gradients():
    B, H, T, d = 1, 2, 8, 4
    Q, K, V, dO = (RNG.normal(size=(B, H, T, d)) for _ in range(4))
    alpha = RNG.normal(size=(H, T))
    rho = -np.log1p(np.arange(T))[None, :] + RNG.normal(0, 0.3, size=(H, T))
    mask = np.array([1, 0], dtype=np.uint8)
    dQ, dK, dV, da, dr = oracle.hybrid_attn_bwd(Q, K, V, alpha, rho, mask, dO)
    f = lambda: _loss(Q, K, V, alpha, rho, mask, dO)
    np.testing.assert_allclose(dQ, _fd(f, Q), rtol=0, atol=2e-8)
    np.testing.assert_allclose(dK, _fd(f, K), rtol=0, atol=2e-8)
    np.testing.assert_allclose(dV, _fd(f, V), rtol=0, atol=2e-8)
    fa = _fd(f, alpha)
    fr = _fd(f, rho)
    np.testing.assert_allclose(da[0], fa[0], rtol=0, atol=2e-8)
    np.testing.assert_allclose(dr[0], fr[0], rtol=0, atol=2e-8)
    # dynamic rows of alpha/rho do not influence the loss and stay zero
    assert np.all(da[1] == 0) and np.all(dr[1] == 0)
    assert np.all(np.abs(fa[1]) < 1e-9) and np.all(np.abs(fr[1]) < 1e-9)
    # static heads get no query/key gradient
    assert np.all(dQ[:, 0] == 0) and np.all(dK[:, 0] == 0)


def test_dynamic_backward_matches_library_autograd():
    T, d = 24, 8
    q, k, v, dO = (RNG.normal(size=(T, d)) for _ in range(4))
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        tq[None, None], tk[None, None], tv[None, None], is_causal=True)[0, 0]
    (out * torch.from_numpy(dO)).sum().backward()
    dq, dk, dv = oracle.dynamic_head_bwd(q, k, v, dO)
    np.testing.assert_allclose(dq, tq.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), atol=1e-12)


def test_gauge_sums_vanish():
    T, d, B = 40, 4, 3
    alpha = RNG.normal(size=T)
    rho = RNG.normal(size=T)
    vs = [RNG.normal(size=(T, d)) for _ in range(B)]
    dos = [RNG.normal(size=(T, d)) for _ in range(B)]
    _, da, dr = oracle.static_head_bwd(alpha, rho, vs, dos)
    scale = np.abs(da).max() + np.abs(dr).max()
    assert abs(da.sum()) < 1e-12 * max(1, scale) * T
    assert abs(dr.sum()) < 1e-12 * max(1, scale) * T


def test_identity_pattern_passes_gradient_through():
    T, d = 16, 3
    rho = np.full(T, -np.inf); rho[0] = 0.0
    dO = RNG.normal(size=(T, d))
    dvs, _, _ = oracle.static_head_bwd(RNG.normal(size=T), rho, [RNG.normal(size=(T, d))], [dO])
    np.testing.assert_allclose(dvs[0], dO, atol=1e-14)


def test_running_mean_pattern_backward_closed_form():
    T, d = 21, 2
    dO = RNG.normal(size=(T, d))
    dvs, _, _ = oracle.static_head_bwd(np.zeros(T), np.zeros(T), [RNG.normal(size=(T, d))], [dO])
    want = np.array([(dO[j:] / np.arange(j + 1, T + 1)[:, None]).sum(0) for j in range(T)])
    np.testing.assert_allclose(dvs[0], want, atol=1e-13)


def test_row_block_parts_sum_to_full_backward():
    T, d = 40, 4
    q, k, v, dO = (RNG.normal(size=(T, d)) for _ in range(4))
    alpha, rho = RNG.normal(size=T), RNG.normal(size=T)
    dq, dk, dv = oracle.dynamic_head_bwd(q, k, v, dO)
    blocks = [range(0, 13), range(13, 31), range(31, 40)]
    parts = [oracle.dynamic_head_bwd_rows(q, k, v, dO, list(b)) for b in blocks]
    np.testing.assert_allclose(np.concatenate([p[0] for p in parts]), dq, atol=1e-13)
    np.testing.assert_allclose(sum(p[1] for p in parts), dk, atol=1e-13)
    np.testing.assert_allclose(sum(p[2] for p in parts), dv, atol=1e-13)
    dvs, da, dr = oracle.static_head_bwd(alpha, rho, [v], [dO])
    parts = [oracle.static_head_bwd_rows(alpha, rho, v, dO, list(b)) for b in blocks]
    np.testing.assert_allclose(sum(p[0] for p in parts), dvs[0], atol=1e-13)
    np.testing.assert_allclose(sum(p[1] for p in parts), da, atol=1e-13)
    np.testing.assert_allclose(sum(p[2] for p in parts), dr, atol=1e-13)
