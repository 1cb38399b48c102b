"""Shared helpers for the parity tests (GPU side marshalling and tolerances).

Tolerance (bf16 outputs and gradients): per tensor and per head class,
    max|x - y| <= 2e-2 * max(1, max|y|)   and   ||x - y||_2 / ||y||_2 <= 1e-2,
with the oracle fed the same bf16-rounded inputs upcast to float64.  For
O(1) tensors this is the plain max-abs 2e-2 / rel-L2 1e-2 bar; for tensors
whose magnitude grows with T or B (dV of early keys, dalpha, drho) the max-abs
bound scales with the tensor's own magnitude, since a bf16 result carries a
relative rounding error of 2^-9 whatever its size.
"""

import numpy as np

ATOL = 2e-2
REL_L2 = 1e-2


def assert_close(got, want, name, atol=ATOL, rel_l2=REL_L2):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - want).max() if got.size else 0.0
    scale = max(1.0, float(np.abs(want).max()) if want.size else 0.0)
    nrm = np.linalg.norm(want)
    rel = np.linalg.norm(got - want) / nrm if nrm > 0 else np.linalg.norm(got - want)
    assert err <= atol * scale, f"{name}: max abs err {err:.3e} > {atol * scale:.3e}"
    assert rel <= rel_l2, f"{name}: rel L2 err {rel:.3e} > {rel_l2:.1e}"
    return err, rel


def bf16_round(x):
    """Round float32/float64 arrays to bf16 and back to float64 (the values
    the GPU sees)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).to(torch.float64).numpy()


def to_dev(x, dtype):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        device="cuda", dtype=dtype)


def to_np(t):
    return t.detach().to("cpu", dtype=__import__("torch").float64).numpy()
