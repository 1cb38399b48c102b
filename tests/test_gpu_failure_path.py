"""The failure path of the kernels' bounded waits, exercised without a GPU fault.

Every mbarrier wait in the attention kernels gives up after a limit: the CTA
then records SAF_ERR_TIMEOUT and a site code in the workspace's status word,
abandons its remaining waits, lets the copies and tensor-core products it
issued finish, frees its tensor memory and returns.  Here one release is
withheld on purpose (saf_debug_forward_hold: the forward's first CTA never
issues its first Q tile), so its waits run out after their 2 s limit.  The test
checks that the launch returns without a CUDA error, that the status word
reports a timeout at a forward site, and that the next forward on the same
workspace runs normally and matches the float64 oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, bf16_round, to_dev, to_np
from dynamic_causal_attention_gb300.synthetic import AttnConfig, attn_inputs

pytestmark = pytest.mark.gpu

FORWARD_SITES = range(1, 15)  # the forward kernel's site codes


def test_withheld_tile_times_out_and_the_context_survives():
    from dynamic_causal_attention_gb300 import _binding as B
    from dynamic_causal_attention_gb300 import api

    # two dynamic heads, T = 256: four items, one per CTA, so that the CTA
    # that withholds its Q tile has nothing else to load
    cfg = AttnConfig("fail", B=1, H=2, T=256, d_h=64, dtype="bf16", static_heads=())
    inp = attn_inputs(cfg, seed=91)
    q, k, v = (to_dev(inp[n], torch.bfloat16) for n in ("Q", "K", "V"))
    alpha = to_dev(inp["alpha"], torch.float32)
    rho = to_dev(inp["rho"], torch.float32)
    layer = api.HybridAttention(cfg.B, cfg.H, cfg.T, cfg.d_h, cfg.head_is_static)

    assert B.saf_debug_forward_hold(1) == B.SAF_OK
    try:
        layer.forward(q, k, v, alpha, rho)
        torch.cuda.synchronize()          # the kernel returned, no CUDA error
        st, site = layer.device_status()
    finally:
        B.saf_debug_forward_hold(0)
    assert st == B.SAF_ERR_TIMEOUT, B.saf_status_string(st)
    assert site in FORWARD_SITES, site

    # the same workspace, normal operation: correct results, clean status
    Q, K, V = (bf16_round(inp[n]) for n in ("Q", "K", "V"))
    ref_out, ref_lse = oracle.hybrid_attn_fwd(Q, K, V, inp["alpha"], inp["rho"],
                                              cfg.head_is_static)
    for _ in range(2):
        out, lse = layer.forward(q, k, v, alpha, rho)
        torch.cuda.synchronize()
        st, site = layer.device_status()
        assert st == B.SAF_OK, (B.saf_status_string(st), site)
        assert_close(to_np(out), ref_out, "out after a timeout")
        assert_close(to_np(lse), ref_lse, "lse after a timeout", atol=1e-3, rel_l2=1e-4)
