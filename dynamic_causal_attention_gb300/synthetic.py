"""Seeded synthetic workloads for the SAF hybrid attention layer and calibration.

This module only draws random numbers and lays them out.  It holds none of
the method's arithmetic: no attention, no fixed pattern, no calibration
statistic.  The calibration inputs are row-stochastic causal matrices made by
the library routine ``torch.softmax`` over random masked logits (the stand-in
for a model's captured attention probabilities); the reduction under test
only consumes them.

Both the CUDA path's tests/bench and the float64 oracle are fed from here.

Workloads (shapes of "When Can Attention Heads Be Statically Defined?",
§4 and Table 2: 124M = 12 layers x 12 heads x 768, T = 4K; 1B at T = 8K):

* ``tiny``  : B=1, H=4 (head 0 static), T=128, d_h=32, fp32 I/O.
              Q, K, V ~ N(0,1); alpha ~ N(0,1); rho(d) = -0.05 d + N(0, 0.5).
* ``124m``  : B=8, H=12, d_h=64, T=4096, bf16; 3 static heads.
              Q, K, V ~ N(0,1); alpha ~ N(0,1); rho(d) = -log(1+d) + N(0, 0.3).
* ``1b``    : B=2, H=16, d_h=128, T=8192, bf16; 4 static heads; same
              distributions as ``124m``; the alpha/rho gradients are requested.
* ``calib`` : N=64 sequences, 12 x 12 = 144 heads, T=1024; probabilities
              softmax_causal(Q K^T / (sqrt(64) tau_h)) with Q, K ~ N(0,1) and a
              per-head temperature tau_h ~ U(0.1, 3); k = round(0.25 * 144).

N(0, s) means standard deviation s.  The upstream gradient dO ~ N(0,1).
Static heads are the first H_s entries of a permutation drawn with seed 0
(``tiny`` fixes head 0).  Draw order from one seeded PCG64 stream:
Q, K, V, alpha, rho noise, dO.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

__all__ = [
    "AttnConfig",
    "CalibConfig",
    "ATTN_CONFIGS",
    "CALIB_CONFIG",
    "static_heads_for_ratio",
    "attn_inputs",
    "calib_temperatures",
    "calib_probabilities",
    "prefill_inputs",
    "PREFILL_SWEEP",
]


@dataclass(frozen=True)
class AttnConfig:
    name: str
    B: int
    H: int
    T: int
    d_h: int
    dtype: str                       # "f32" or "bf16": the I/O type
    static_heads: tuple = ()
    dist: str = "124m"               # "tiny" or "124m" value distributions
    want_param_grads: bool = False
    extra: dict = field(default_factory=dict)

    @property
    def head_is_static(self) -> np.ndarray:
        m = np.zeros(self.H, dtype=np.uint8)
        for h in self.static_heads:
            m[h] = 1
        return m


def static_heads_for_ratio(H: int, r: float, seed: int = 0) -> tuple:
    """The first round(r H) heads (half to even) of a seeded permutation."""
    k = int(round(r * H))
    perm = np.random.default_rng(seed).permutation(H)
    return tuple(sorted(int(h) for h in perm[:k]))


ATTN_CONFIGS = {
    "tiny": AttnConfig("tiny", B=1, H=4, T=128, d_h=32, dtype="f32",
                       static_heads=(0,), dist="tiny"),
    "124m": AttnConfig("124m", B=8, H=12, T=4096, d_h=64, dtype="bf16",
                       static_heads=static_heads_for_ratio(12, 0.25)),
    "1b": AttnConfig("1b", B=2, H=16, T=8192, d_h=128, dtype="bf16",
                     static_heads=static_heads_for_ratio(16, 0.25),
                     want_param_grads=True),
}


def sweep_config(r: float) -> AttnConfig:
    """The 124M-shaped layer with a fraction r of its heads static."""
    base = ATTN_CONFIGS["124m"]
    return replace(base, name=f"124m_r{r:g}",
                   static_heads=static_heads_for_ratio(base.H, r))


def attn_inputs(cfg: AttnConfig, seed: int = 0, **shape_overrides):
    """Draw Q, K, V, alpha, rho, dO for ``cfg`` as float32 NumPy arrays.

    ``shape_overrides`` (B, H, T, d_h) shrink a workload for parity tests
    while keeping its value distributions.
    """
    B = shape_overrides.get("B", cfg.B)
    H = shape_overrides.get("H", cfg.H)
    T = shape_overrides.get("T", cfg.T)
    d = shape_overrides.get("d_h", cfg.d_h)
    rng = np.random.Generator(np.random.PCG64(seed))
    shp = (B, H, T, d)
    Q = rng.standard_normal(shp, dtype=np.float32)
    K = rng.standard_normal(shp, dtype=np.float32)
    V = rng.standard_normal(shp, dtype=np.float32)
    alpha = rng.standard_normal((H, T), dtype=np.float32)
    delta = np.arange(T, dtype=np.float64)
    if cfg.dist == "tiny":
        noise = rng.normal(0.0, 0.5, size=(H, T))
        rho = (-0.05 * delta)[None, :] + noise
    else:
        noise = rng.normal(0.0, 0.3, size=(H, T))
        rho = (-np.log1p(delta))[None, :] + noise
    rho = rho.astype(np.float32)
    dO = rng.standard_normal(shp, dtype=np.float32)
    return {"Q": Q, "K": K, "V": V, "alpha": alpha, "rho": rho, "dO": dO}


@dataclass(frozen=True)
class CalibConfig:
    name: str = "calib"
    N: int = 64
    L: int = 12
    H: int = 12
    T: int = 1024
    d_h: int = 64
    r: float = 0.25

    @property
    def num_heads(self) -> int:
        return self.L * self.H


CALIB_CONFIG = CalibConfig()


def calib_temperatures(num_heads: int, seed: int = 0) -> np.ndarray:
    """tau_h ~ U(0.1, 3), drawn once per head."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    return rng.uniform(0.1, 3.0, size=num_heads)


def calib_probabilities(N: int, num_heads: int, T: int, d_h: int = 64,
                        seed: int = 0, device: str = "cpu", out=None,
                        n_begin: int = 0, n_count: int | None = None,
                        want_logits: bool = False):
    """Row-stochastic causal probability matrices, float32 [n, heads, T, T].

    Sample n of head h is torch.softmax over Q K^T / (sqrt(d_h) tau_h) with
    -inf above the diagonal, where Q, K ~ N(0,1) are drawn from a torch
    generator seeded with (seed, n).  Returns a torch tensor on ``device``
    (written into ``out`` when given).  ``n_begin``/``n_count`` select a
    slice of the N samples so that callers can stream them.  With
    ``want_logits`` the pre-softmax logits are returned instead, zero above
    the diagonal.
    """
    import torch

    if n_count is None:
        n_count = N - n_begin
    tau = torch.tensor(calib_temperatures(num_heads, seed), dtype=torch.float32,
                       device=device)
    scale = 1.0 / (np.sqrt(d_h) * tau)                     # [heads]
    if out is None:
        out = torch.empty((n_count, num_heads, T, T), dtype=torch.float32,
                          device=device)
    mask = torch.ones((T, T), dtype=torch.bool, device=device).triu(1)
    for n in range(n_begin, n_begin + n_count):
        g = torch.Generator(device=device)
        g.manual_seed(int(seed) * 1_000_003 + n)
        q = torch.randn((num_heads, T, d_h), generator=g, device=device)
        k = torch.randn((num_heads, T, d_h), generator=g, device=device)
        logits = torch.matmul(q, k.transpose(1, 2)) * scale[:, None, None]
        if want_logits:
            out[n - n_begin] = logits.masked_fill_(mask, 0.0)
        else:
            logits.masked_fill_(mask, float("-inf"))
            out[n - n_begin] = torch.softmax(logits, dim=-1)
        del q, k, logits
    return out


# Forward-only causal prefill sweep (App. D.3 of the notes: the 124M model's
# head shape, batch 64, T from 512 to 16K, 25% and 50% of heads frozen, plus
# batch 1 at T = 4096 where launch overhead dominates).
PREFILL_SWEEP = {
    "B": 64, "H": 12, "d_h": 64,
    "T": (512, 1024, 2048, 4096, 8192, 16384),
    "ratios": (0.0, 0.25, 0.5),
    "batch1_T": 4096,
}


def prefill_inputs(B: int, H: int, T: int, d_h: int, seed: int = 0, device: str = "cuda"):
    """Q, K, V ~ N(0,1) as bf16 device tensors drawn with a seeded torch
    generator on ``device`` (large prefill shapes are drawn where they are
    used), and alpha ~ N(0,1), rho(d) = -log(1+d) + N(0, 0.3) as fp32."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed) * 7919 + T)
    shp = (B, H, T, d_h)
    q = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(shp, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    rng = np.random.Generator(np.random.PCG64(seed + T))
    alpha = rng.standard_normal((H, T), dtype=np.float32)
    rho = (-np.log1p(np.arange(T, dtype=np.float64))[None, :]
           + rng.normal(0.0, 0.3, size=(H, T))).astype(np.float32)
    return q, k, v, torch.from_numpy(alpha).to(device), torch.from_numpy(rho).to(device)
