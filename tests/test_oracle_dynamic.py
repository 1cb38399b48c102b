"""Pins for the oracle's dynamic (ordinary causal softmax) head."""

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(99)


def test_golden_dynamic_head(golden):
    g = golden("dynamic_head_T2.txt")
    q, k, v = (g[n][:, None] for n in ("q", "k", "v"))
    out, lse, A = oracle.dynamic_head_fwd(q, k, v)
    np.testing.assert_allclose(A, g["A"], atol=1e-15)
    np.testing.assert_allclose(out[:, 0], g["O"], atol=1e-14)
    np.testing.assert_allclose(lse, g["lse"], atol=1e-14)


def test_zero_query_gives_running_mean():
    T, d = 30, 6
    v = RNG.normal(size=(T, d))
    out, lse, _ = oracle.dynamic_head_fwd(np.zeros((T, d)), RNG.normal(size=(T, d)), v)
    np.testing.assert_allclose(out, np.cumsum(v, 0) / np.arange(1, T + 1)[:, None], atol=1e-13)
    np.testing.assert_allclose(lse, np.log(np.arange(1, T + 1)), atol=1e-13)


@pytest.mark.parametrize("T,d", [(1, 4), (17, 8), (64, 32)])
def test_matches_library_sdpa_float64(T, d):
    q, k, v = (RNG.normal(size=(T, d)) for _ in range(3))
    out, lse, A = oracle.dynamic_head_fwd(q, k, v)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None], torch.from_numpy(k)[None, None],
        torch.from_numpy(v)[None, None], is_causal=True)[0, 0].numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # lse against the library's logsumexp of the masked scores
    s = torch.from_numpy(q @ k.T / np.sqrt(d))
    s = s.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=1).numpy(), atol=1e-12)
    np.testing.assert_allclose(A.sum(1), 1.0, atol=1e-12)
    assert np.all(A[np.triu_indices(T, 1)] == 0)
