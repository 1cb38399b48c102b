"""Parity at sequence lengths that are not a multiple of 128, and at the most
heads a call takes.

The kernels work on whole 128-row tiles; the C ABI runs such a length on
zero-padded copies in the workspace (alpha and rho padded with -inf, the
padded rows' lse 0) and crops the results.  Every output and gradient of the
real rows must equal the float64 oracle at length T, whatever the padding
holds: lengths of one row, of a few rows, just past a tile edge and inside a
later tile, with frozen heads (factored and exact generator modes), grouped
K/V and fp32 I/O.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, bf16_round, to_dev, to_np
from dynamic_causal_attention_gb300.synthetic import AttnConfig, attn_inputs

pytestmark = pytest.mark.gpu


def run(inp, mask, grads, dtype=torch.bfloat16, H_kv=None):
    from dynamic_causal_attention_gb300 import api
    B, H, T, d = inp["V"].shape
    Hkv = H if H_kv is None else H_kv
    layer = api.HybridAttention(B, H, T, d, mask, dtype=dtype, want_param_grads=grads, H_kv=Hkv)
    q = to_dev(inp["Q"], dtype)
    k = to_dev(inp["K"][:, :Hkv], dtype)
    v = to_dev(inp["V"][:, :Hkv], dtype)
    do = to_dev(inp["dO"], dtype)
    alpha = to_dev(inp["alpha"], torch.float32)
    rho = to_dev(inp["rho"], torch.float32)
    out, lse = layer.forward(q, k, v, alpha, rho)
    torch.cuda.synchronize()
    st, site = layer.device_status()
    assert st == 0, f"forward: wait timed out at site {site}"
    res = layer.backward(q, k, v, out, lse, do, alpha, rho, want_param_grads=grads)
    torch.cuda.synchronize()
    st, site = layer.device_status()
    assert st == 0, f"backward: wait timed out at site {site}"
    return [to_np(out), to_np(lse)] + [None if x is None else to_np(x) for x in res]


def check(cfg, inp, got, grads, H_kv=None):
    st = np.asarray(cfg.head_is_static, bool)
    Hkv = cfg.H if H_kv is None else H_kv
    Q, dO = bf16_round(inp["Q"]), bf16_round(inp["dO"])
    K, V = bf16_round(inp["K"][:, :Hkv]), bf16_round(inp["V"][:, :Hkv])
    if H_kv is None:
        ref_out, ref_lse = oracle.hybrid_attn_fwd(Q, K, V, inp["alpha"], inp["rho"],
                                                  cfg.head_is_static)
        rq, rk, rv, ra, rr = oracle.hybrid_attn_bwd(Q, K, V, inp["alpha"], inp["rho"],
                                                    cfg.head_is_static, dO, grads)
    else:
        ref_out, ref_lse = oracle.gqa_hybrid_attn_fwd(Q, K, V, inp["alpha"], inp["rho"],
                                                      cfg.head_is_static)
        rq, rk, rv, ra, rr = oracle.gqa_hybrid_attn_bwd(Q, K, V, inp["alpha"], inp["rho"],
                                                        cfg.head_is_static, dO, grads)
    out, lse, dq, dk, dv, da, dr = got
    tag = f"T={cfg.T} d={cfg.d_h}"
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    for cls, sel in (("static", st), ("dynamic", ~st)):
        if sel.any():
            assert_close(out[:, sel], ref_out[:, sel], f"{tag} out[{cls}]")
            assert_close(lse[:, sel], ref_lse[:, sel], f"{tag} lse[{cls}]", atol=1e-3, rel_l2=1e-4)
    if (~st).any():
        assert_close(dq[:, ~st], rq[:, ~st], f"{tag} dQ")
    assert np.all(dq[:, st] == 0)
    assert_close(dk, rk, f"{tag} dK")
    assert_close(dv, rv, f"{tag} dV")
    if grads and st.any():
        assert_close(da[st], ra[st], f"{tag} dalpha")
        assert_close(dr[st], rr[st], f"{tag} drho")


@pytest.mark.parametrize("T,d_h", [(1, 64), (5, 32), (100, 64), (129, 128), (200, 64),
                                   (333, 32), (383, 128)])
def test_ragged_length_matches_oracle(T, d_h):
    cfg = AttnConfig("ragged", B=2, H=4, T=T, d_h=d_h, dtype="bf16", static_heads=(1, 2))
    inp = attn_inputs(cfg, seed=300 + T)
    check(cfg, inp, run(inp, cfg.head_is_static, True), True)


def test_ragged_length_exact_mode_and_fp32():
    # a frozen head whose parameter range needs the exact exponential, fp32 I/O
    cfg = AttnConfig("ragged_x", B=2, H=3, T=250, d_h=64, dtype="f32", static_heads=(0, 2))
    inp = attn_inputs(cfg, seed=311)
    inp["alpha"][0] = (0.45 * np.arange(cfg.T) - 60.0).astype(np.float32)
    check(cfg, inp, run(inp, cfg.head_is_static, True, dtype=torch.float32), True)


def test_ragged_length_grouped_kv():
    cfg = AttnConfig("ragged_g", B=2, H=4, T=170, d_h=64, dtype="bf16", static_heads=(1,))
    inp = attn_inputs(cfg, seed=313)
    check(cfg, inp, run(inp, cfg.head_is_static, True, H_kv=2), True, H_kv=2)


def test_most_heads_at_once():
    # H = 256, the most heads a call takes (one item per head and sequence),
    # a third of them frozen, with the head index stored in 8 bits everywhere
    H = 256
    static = tuple(range(0, H, 3))
    cfg = AttnConfig("many_heads", B=1, H=H, T=128, d_h=32, dtype="bf16", static_heads=static)
    inp = attn_inputs(cfg, seed=317)
    check(cfg, inp, run(inp, cfg.head_is_static, True), True)
