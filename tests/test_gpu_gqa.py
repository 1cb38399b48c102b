"""Parity of grouped K/V (the GQA path: K/V shared by groups of query heads,
a frozen query head still mixing its group's V) with the float64 grouped
oracle, forward and backward, through the C ABI.  The groups mix frozen and
dynamic query heads, hold only frozen or only dynamic ones, and shrink to a
single K/V head (MQA)."""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, bf16_round, to_dev, to_np
from dynamic_causal_attention_gb300.synthetic import AttnConfig, attn_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    from dynamic_causal_attention_gb300 import api as _api
    return _api


def gqa_inputs(B, H, H_kv, T, d, static, seed):
    cfg = AttnConfig("gqa", B=B, H=H, T=T, d_h=d, dtype="bf16", static_heads=static)
    inp = attn_inputs(cfg, seed=seed)
    inp["K"] = np.ascontiguousarray(inp["K"][:, :H_kv])
    inp["V"] = np.ascontiguousarray(inp["V"][:, :H_kv])
    return cfg, inp


def run(api, cfg, inp, H_kv, grads, dtype=torch.bfloat16):
    B, H, T, d = inp["Q"].shape
    layer = api.HybridAttention(B, H, T, d, cfg.head_is_static, dtype=dtype,
                                want_param_grads=grads, H_kv=H_kv)
    q, k, v, do = (to_dev(inp[n], dtype) for n in ("Q", "K", "V", "dO"))
    alpha = to_dev(inp["alpha"], torch.float32)
    rho = to_dev(inp["rho"], torch.float32)
    out, lse = layer.forward(q, k, v, alpha, rho)
    res = layer.backward(q, k, v, out, lse, do, alpha, rho, want_param_grads=grads)
    torch.cuda.synchronize()
    st, site = layer.device_status()
    assert st == 0, f"device wait timed out at site {site}"
    return [to_np(out), to_np(lse)] + [None if x is None else to_np(x) for x in res]


def check(got, inp, mask, grads, tag):
    Q, K, V, dO = (bf16_round(inp[n]) for n in ("Q", "K", "V", "dO"))
    ro, rl = oracle.gqa_hybrid_attn_fwd(Q, K, V, inp["alpha"], inp["rho"], mask)
    rq, rk, rv, ra, rr = oracle.gqa_hybrid_attn_bwd(Q, K, V, inp["alpha"], inp["rho"], mask, dO,
                                                    grads)
    out, lse, dq, dk, dv, da, dr = got
    st = np.asarray(mask, bool)
    assert_close(out, ro, f"{tag} out")
    np.testing.assert_allclose(lse, rl, atol=1e-3, err_msg=f"{tag} lse")
    if (~st).any():
        assert_close(dq[:, ~st], rq[:, ~st], f"{tag} dQ")
    assert np.all(dq[:, st] == 0)
    assert_close(dk, rk, f"{tag} dK")
    assert_close(dv, rv, f"{tag} dV")
    if grads:
        assert_close(da[st], ra[st], f"{tag} dalpha")
        assert_close(dr[st], rr[st], f"{tag} drho")


@pytest.mark.parametrize("d_h", [32, 64, 128])
@pytest.mark.parametrize("B,H,H_kv,T,static,grads", [
    (2, 8, 2, 384, (1, 2, 5), True),        # every group mixes frozen and dynamic heads
    (1, 8, 4, 256, (2, 3, 4), False),       # one group all frozen, two all dynamic, one mixed
    (2, 4, 1, 256, (1,), False),            # a single K/V head for all query heads
])
def test_gqa_matches_oracle(api, d_h, B, H, H_kv, T, static, grads):
    cfg, inp = gqa_inputs(B, H, H_kv, T, d_h, static, seed=61 + d_h)
    got = run(api, cfg, inp, H_kv, grads)
    check(got, inp, cfg.head_is_static, grads, f"gqa d{d_h} H{H}/{H_kv}")


def test_gqa_many_items_per_cta(api):
    cfg, inp = gqa_inputs(8, 12, 4, 512, 64, (2, 7, 9), seed=67)
    got = run(api, cfg, inp, 4, True)
    check(got, inp, cfg.head_is_static, True, "gqa many")


def test_gqa_fp32_io(api):
    cfg, inp = gqa_inputs(1, 4, 2, 128, 32, (0,), seed=71)
    got = run(api, cfg, inp, 2, True, dtype=torch.float32)
    check(got, inp, cfg.head_is_static, True, "gqa fp32")


def test_gqa_exact_range_frozen_head(api):
    # a frozen query head whose alpha spans more than 80 uses the exact
    # exponential; its group mixes it with dynamic heads
    cfg, inp = gqa_inputs(2, 4, 2, 256, 64, (1, 2), seed=73)
    inp["alpha"][1] += np.linspace(-45.0, 45.0, 256)
    got = run(api, cfg, inp, 2, True)
    check(got, inp, cfg.head_is_static, True, "gqa exact")


def test_gqa_no_alloc_forward_matches(api):
    # the allocation-free forward reads grouped K/V the same way
    from dynamic_causal_attention_gb300 import _binding as B
    cfg, inp = gqa_inputs(2, 8, 2, 256, 64, (1, 6), seed=79)
    Bn, H, T, d = inp["Q"].shape
    layer = api.HybridAttention(Bn, H, T, d, cfg.head_is_static, H_kv=2)
    q, k, v = (to_dev(inp[n], torch.bfloat16) for n in ("Q", "K", "V"))
    alpha = to_dev(inp["alpha"], torch.float32)
    rho = to_dev(inp["rho"], torch.float32)
    out, lse = layer.forward(q, k, v, alpha, rho)
    out2 = torch.empty_like(out)
    lse2 = torch.empty_like(lse)
    st = B.saf_hybrid_attn_fwd_noalloc(layer.dims, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                       alpha.data_ptr(), rho.data_ptr(), layer.head_is_static,
                                       out2.data_ptr(), lse2.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
