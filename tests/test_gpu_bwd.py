"""Parity of the hybrid layer's backward (libsaf, sm_103a) with the float64
oracle: dQ, dK, dV for dynamic heads, dV (and optionally dalpha, drho) for
frozen heads, zero dQ/dK on frozen heads.  Same inputs and tolerance rules as
the forward tests; the backward is fed the GPU's own forward output and lse
(as in training), while the oracle recomputes everything from the inputs.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, bf16_round, to_dev, to_np
from dynamic_causal_attention_gb300.synthetic import ATTN_CONFIGS, AttnConfig, attn_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from dynamic_causal_attention_gb300 import api as _api
    return _api


def gpu_fwd_bwd(api, inp, mask, grads, dtype=torch.bfloat16):
    B, H, T, d = inp["V"].shape
    layer = api.HybridAttention(B, H, T, d, mask, dtype=dtype, want_param_grads=grads)
    q, k, v, do = (to_dev(inp[n], dtype) for n in ("Q", "K", "V", "dO"))
    alpha = to_dev(inp["alpha"], torch.float32)
    rho = to_dev(inp["rho"], torch.float32)
    out, lse = layer.forward(q, k, v, alpha, rho)
    torch.cuda.synchronize()
    st, site = layer.device_status()
    assert st == 0, f"forward: device wait timed out at site {site}"
    res = layer.backward(q, k, v, out, lse, do, alpha, rho, want_param_grads=grads)
    torch.cuda.synchronize()
    st, site = layer.device_status()
    assert st == 0, f"device wait timed out at site {site}"
    return [None if x is None else to_np(x) for x in res]


def oracle_bwd(inp, mask, grads):
    Q, K, V, dO = (bf16_round(inp[n]) for n in ("Q", "K", "V", "dO"))
    return oracle.hybrid_attn_bwd(Q, K, V, inp["alpha"], inp["rho"], mask, dO, grads)


def compare(got, ref, mask, tag, grads):
    st = np.asarray(mask, bool)
    dq, dk, dv, da, dr = got
    rq, rk, rv, ra, rr = ref
    if (~st).any():
        assert_close(dq[:, ~st], rq[:, ~st], f"{tag} dQ")
        assert_close(dk[:, ~st], rk[:, ~st], f"{tag} dK")
        assert_close(dv[:, ~st], rv[:, ~st], f"{tag} dV[dynamic]")
    if st.any():
        assert np.all(dq[:, st] == 0) and np.all(dk[:, st] == 0)
        assert_close(dv[:, st], rv[:, st], f"{tag} dV[static]")
        if grads:
            assert_close(da[st], ra[st], f"{tag} dalpha")
            assert_close(dr[st], rr[st], f"{tag} drho")
    if grads:
        assert np.all(da[~st] == 0) and np.all(dr[~st] == 0)


def test_tiny_config_fp32_with_param_grads(api):
    cfg = ATTN_CONFIGS["tiny"]
    inp = attn_inputs(cfg)
    got = gpu_fwd_bwd(api, inp, cfg.head_is_static, True, dtype=torch.float32)
    compare(got, oracle_bwd(inp, cfg.head_is_static, True), cfg.head_is_static, "tiny", True)


@pytest.mark.parametrize("d_h", [32, 64, 128])
@pytest.mark.parametrize("B,H,T,static,grads", [(2, 3, 384, (1,), True), (1, 2, 256, (), False),
                                                (3, 2, 256, (0, 1), True),
                                                (2, 4, 640, (0, 3), False)])
def test_hybrid_bwd_matches_oracle(api, d_h, B, H, T, static, grads):
    cfg = AttnConfig("t", B=B, H=H, T=T, d_h=d_h, dtype="bf16", static_heads=static)
    inp = attn_inputs(cfg, seed=21 + d_h)
    got = gpu_fwd_bwd(api, inp, cfg.head_is_static, grads)
    compare(got, oracle_bwd(inp, cfg.head_is_static, grads), cfg.head_is_static, f"d{d_h}", grads)


@pytest.mark.parametrize("d_h,grads", [(64, False), (128, True)])
def test_many_items_per_cta(api, d_h, grads):
    # More work items than SMs in every kernel of the backward.
    cfg = AttnConfig("many", B=8, H=12, T=512, d_h=d_h, dtype="bf16",
                     static_heads=(2, 7, 9))
    inp = attn_inputs(cfg, seed=43)
    got = gpu_fwd_bwd(api, inp, cfg.head_is_static, grads)
    compare(got, oracle_bwd(inp, cfg.head_is_static, grads), cfg.head_is_static,
            f"many d{d_h}", grads)


@pytest.mark.parametrize("d_h,static,grads", [(64, (), False), (64, (1, 4, 6, 9, 10, 11), False),
                                             (128, (1, 4, 6, 9, 10, 11), True)])
def test_many_short_odd_items(api, d_h, static, grads):
    # Tens of short items per persistent CTA in every kernel (T = 640: key
    # tiles of 1..5 query tiles each, many of odd length), with and without
    # frozen heads, so every item-boundary hand-over repeats many times.
    cfg = AttnConfig("short", B=16, H=12, T=640, d_h=d_h, dtype="bf16", static_heads=static)
    inp = attn_inputs(cfg, seed=47)
    got = gpu_fwd_bwd(api, inp, cfg.head_is_static, grads)
    compare(got, oracle_bwd(inp, cfg.head_is_static, grads), cfg.head_is_static,
            f"short d{d_h}", grads)


@pytest.mark.parametrize("d_h", [64, 128])
def test_backward_run_to_run(api, d_h):
    # Two backward passes on the same inputs.  dK and dV accumulate in tensor
    # memory in a fixed order (and the frozen heads' dV comes from the
    # transposed forward engine, which has no atomics): bit for bit equal.
    # dQ is summed over key tiles by fp32 reduce-adds in whatever order the
    # CTAs arrive, and dalpha/drho by fp32 atomics: the two runs may differ
    # by the rounding of a reordered fp32 sum, which after the bf16
    # conversion of dQ is at most one bf16 unit in the last place.
    cfg = AttnConfig("rep", B=16, H=12, T=640, d_h=d_h, dtype="bf16",
                     static_heads=(1, 4, 6, 9, 10, 11))
    inp = attn_inputs(cfg, seed=49)
    a = gpu_fwd_bwd(api, inp, cfg.head_is_static, True)
    b = gpu_fwd_bwd(api, inp, cfg.head_is_static, True)
    np.testing.assert_array_equal(a[1], b[1])   # dK
    np.testing.assert_array_equal(a[2], b[2])   # dV
    dq1, dq2 = a[0], b[0]
    one_ulp = 2.0 ** -7 * np.maximum(np.abs(dq1), np.abs(dq2))
    spread = np.abs(dq1 - dq2)
    assert np.all(spread <= one_ulp + 1e-6 * np.abs(dq1).max()), spread.max()
    for name, x, y in (("dalpha", a[3], b[3]), ("drho", a[4], b[4])):
        st = np.asarray(cfg.head_is_static, bool)
        assert np.abs(x[st] - y[st]).max() <= 1e-5 * np.abs(x[st]).max(), name


def test_identity_pattern_backward(api):
    B, H, T, d = 2, 1, 256, 64
    cfg = AttnConfig("id", B=B, H=H, T=T, d_h=d, dtype="bf16", static_heads=(0,))
    inp = attn_inputs(cfg, seed=6)
    inp["rho"][:] = -np.inf
    inp["rho"][:, 0] = 0.0
    dq, dk, dv, da, dr = gpu_fwd_bwd(api, inp, cfg.head_is_static, True)
    np.testing.assert_array_equal(dv, bf16_round(inp["dO"]))
    # the identity pattern has no free logits: every gradient of alpha/rho is 0
    assert np.abs(da).max() < 1e-4 and np.abs(dr).max() < 1e-4


def test_running_mean_backward_and_gauge(api):
    B, H, T, d = 3, 1, 384, 32
    cfg = AttnConfig("rm", B=B, H=H, T=T, d_h=d, dtype="bf16", static_heads=(0,))
    inp = attn_inputs(cfg, seed=7)
    inp["alpha"][:] = 0.0
    inp["rho"][:] = 0.0
    dq, dk, dv, da, dr = gpu_fwd_bwd(api, inp, cfg.head_is_static, True)
    dO = bf16_round(inp["dO"])[:, 0]
    want = np.cumsum((dO / np.arange(1, T + 1)[None, :, None])[:, ::-1], axis=1)[:, ::-1]
    assert_close(dv[:, 0], want, "running-mean dV")
    # gauge invariance: alpha + c and rho + c leave P unchanged
    scale = np.abs(da).max() + np.abs(dr).max()
    assert abs(da.sum()) <= 1e-3 * scale * np.sqrt(T)
    assert abs(dr.sum()) <= 1e-3 * scale * np.sqrt(T)


@pytest.mark.parametrize("name", ["124m", "1b"])
def test_full_size_one_head_of_each_class(api, name):
    cfg = ATTN_CONFIGS[name]
    inp = attn_inputs(cfg)
    grads = cfg.want_param_grads
    dq, dk, dv, da, dr = gpu_fwd_bwd(api, inp, cfg.head_is_static, grads)
    st = cfg.head_is_static
    hd = [h for h in range(cfg.H) if not st[h]][0]
    hs = cfg.static_heads[0]
    b = cfg.B - 1
    Q, K, V, dO = (bf16_round(inp[n][b, hd]) for n in ("Q", "K", "V", "dO"))
    rq, rk, rv = oracle.dynamic_head_bwd(Q, K, V, dO)
    assert_close(dq[b, hd], rq, f"{name} dQ")
    assert_close(dk[b, hd], rk, f"{name} dK")
    assert_close(dv[b, hd], rv, f"{name} dV[dynamic]")
    vs = [bf16_round(inp["V"][bb, hs]) for bb in range(cfg.B)]
    dos = [bf16_round(inp["dO"][bb, hs]) for bb in range(cfg.B)]
    rvs, ra, rr = oracle.static_head_bwd(inp["alpha"][hs], inp["rho"][hs], vs, dos)
    for bb in range(cfg.B):
        assert_close(dv[bb, hs], rvs[bb], f"{name} dV[static] b{bb}")
    assert np.all(dq[:, hs] == 0) and np.all(dk[:, hs] == 0)
    if grads:
        assert_close(da[hs], ra, f"{name} dalpha")
        assert_close(dr[hs], rr, f"{name} drho")


def test_param_grads_several_rounds_both_generator_modes(api):
    # More (head, key tile) items than SMs, so each CTA takes items from
    # several rounds of the snake order; heads 0 and 5 have a parameter range
    # above 80 and use the exact exponential, the others the factored form.
    B, H, T, d = 1, 8, 2560, 32
    cfg = AttnConfig("rounds", B=B, H=H, T=T, d_h=d, dtype="bf16",
                     static_heads=tuple(range(H)))
    inp = attn_inputs(cfg, seed=57)
    for h in (0, 5):
        inp["alpha"][h] += np.linspace(-45.0, 45.0, T)
    got = gpu_fwd_bwd(api, inp, cfg.head_is_static, True)
    compare(got, oracle_bwd(inp, cfg.head_is_static, True), cfg.head_is_static, "rounds", True)


def test_masked_keys_and_fully_masked_head(api):
    # head 0: alpha = -inf everywhere (no row has a distribution: out = 0,
    # lse = -inf, zero gradients); head 1: every even key masked, so row 0 is
    # empty and the other rows see only odd keys
    B, H, T, d = 2, 2, 256, 64
    cfg = AttnConfig("mask", B=B, H=H, T=T, d_h=d, dtype="bf16", static_heads=(0, 1))
    inp = attn_inputs(cfg, seed=13)
    inp["alpha"][0] = -np.inf
    inp["alpha"][1, 0::2] = -np.inf
    layer = api.HybridAttention(B, H, T, d, cfg.head_is_static, want_param_grads=True)
    q, k, v, do = (to_dev(inp[n], torch.bfloat16) for n in ("Q", "K", "V", "dO"))
    alpha = to_dev(inp["alpha"], torch.float32)
    rho = to_dev(inp["rho"], torch.float32)
    out, lse = layer.forward(q, k, v, alpha, rho)
    dq, dk, dv, da, dr = layer.backward(q, k, v, out, lse, do, alpha, rho, want_param_grads=True)
    torch.cuda.synchronize()
    out, lse, dv, da, dr = (to_np(x) for x in (out, lse, dv, da, dr))
    assert np.all(out[:, 0] == 0) and np.all(np.isneginf(lse[:, 0]))
    assert np.all(out[:, 1, 0] == 0) and np.all(np.isneginf(lse[:, 1, 0]))
    V, dO = bf16_round(inp["V"]), bf16_round(inp["dO"])
    ro, rl = oracle.hybrid_attn_fwd(inp["Q"], inp["K"], V, inp["alpha"], inp["rho"],
                                    cfg.head_is_static)
    assert_close(out[:, 1], ro[:, 1], "masked-keys out")
    np.testing.assert_allclose(lse[:, 1, 1:], rl[:, 1, 1:], atol=1e-3)
    rv, ra, rr = oracle.static_head_bwd(inp["alpha"][1], inp["rho"][1], [V[b, 1] for b in range(B)],
                                        [dO[b, 1] for b in range(B)])
    for b in range(B):
        assert_close(dv[b, 1], rv[b], f"masked-keys dV b{b}")
    assert np.all(dv[:, 0] == 0)
    assert np.all(np.isfinite(da)) and np.all(np.isfinite(dr))
    assert np.all(da[0] == 0) and np.all(dr[0] == 0)
    assert np.all(da[1][0::2] == 0)
    assert_close(da[1][1::2], ra[1::2], "masked-keys dalpha")
    assert_close(dr[1], rr, "masked-keys drho")
