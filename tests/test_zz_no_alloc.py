"""The workspace-free forward entry point, checked against the regular one and
against the oracle.

saf_hybrid_attn_fwd_noalloc is for callers that cannot allocate device memory
while they run the layer, such as an engine plugin that is handed only its
input and output buffers because the engine planned all memory in advance.
Its scratch is one fixed device array inside the library, shared by every call
and keeping the last call's contents, so the tests make calls in a row on
different inputs (a frozen head whose parameter range needs the exact
exponential, then factored ones) and compare each with saf_hybrid_attn_fwd,
which uses a caller-provided workspace, on the same inputs.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run alone.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, bf16_round, to_dev, to_np
from dynamic_causal_attention_gb300.synthetic import AttnConfig, attn_inputs

pytestmark = pytest.mark.gpu

# Shapes either side of the scratch limit (4 MiB): 15 frozen heads fit at
# T = 16384, 16 do not; 16 fit at T = 16256.
LIMIT_OK = (15, 16384)
LIMIT_OK2 = (16, 16256)
LIMIT_OVER = (16, 16384)


def _call_noalloc(B, layer, q, k, v, alpha, rho, out, lse):
    stream = torch.cuda.current_stream().cuda_stream
    p = lambda t: None if t is None else t.data_ptr()
    return B.saf_hybrid_attn_fwd_noalloc(layer.dims, p(q), p(k), p(v), p(alpha), p(rho),
                                         layer.head_is_static, p(out), p(lse), stream)


def _run_pair(cfg, inp, want_lse=True, H_kv=None):
    """(noalloc out, noalloc lse, workspace out, workspace lse) on the same inputs."""
    from dynamic_causal_attention_gb300 import _binding as B
    from dynamic_causal_attention_gb300 import api

    Hkv = cfg.H if H_kv is None else H_kv
    q = to_dev(inp["Q"], torch.bfloat16)
    k = to_dev(inp["K"][:, :Hkv], torch.bfloat16)
    v = to_dev(inp["V"][:, :Hkv], torch.bfloat16)
    alpha = to_dev(inp["alpha"], torch.float32)
    rho = to_dev(inp["rho"], torch.float32)
    layer = api.HybridAttention(cfg.B, cfg.H, cfg.T, cfg.d_h, cfg.head_is_static, H_kv=Hkv)
    ref_out, ref_lse = layer.forward(q, k, v, alpha, rho)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan")) if want_lse else None
    st = _call_noalloc(B, layer, q, k, v, alpha, rho, out, lse)
    assert st == B.SAF_OK, B.saf_status_string(st)
    torch.cuda.synchronize()
    return (to_np(out), None if lse is None else to_np(lse), to_np(ref_out), to_np(ref_lse))


def test_noalloc_forward_matches_workspace_forward_twice():
    cfg = AttnConfig("noalloc", B=2, H=6, T=512, d_h=64, dtype="bf16", static_heads=(1, 4))
    for call, seed in enumerate((51, 52)):
        inp = attn_inputs(cfg, seed=seed)
        if call == 1:
            # a different pattern on the second call: stale tables would show
            inp["alpha"] *= 2.0
            inp["rho"] = (inp["rho"] * 0.5).astype(np.float32)
        out, lse, ref_out, ref_lse = _run_pair(cfg, inp)
        assert_close(out, ref_out, f"call {call} out")
        assert_close(lse, ref_lse, f"call {call} lse", atol=1e-3, rel_l2=1e-4)


@pytest.mark.parametrize("d_h,H_kv", [(32, None), (128, None), (64, 2)])
def test_noalloc_exact_then_factored(d_h, H_kv):
    # First call: frozen head 0 has range(alpha) + range(rho) > 80, so its
    # tables hold log2 values and -inf padding (exact exponential).  Second
    # call: the same head factored.  Both against the workspace forward; the
    # second without lse (the output must not depend on it).
    B, H, T = 3, 4, 384
    cfg = AttnConfig("noalloc_x", B=B, H=H, T=T, d_h=d_h, dtype="bf16", static_heads=(0, 3))
    inp = attn_inputs(cfg, seed=61)
    inp["alpha"][0] = (0.45 * np.arange(T) - 80.0).astype(np.float32)
    out, lse, ref_out, ref_lse = _run_pair(cfg, inp, H_kv=H_kv)
    assert_close(out, ref_out, "exact call out")
    assert_close(lse, ref_lse, "exact call lse", atol=1e-3, rel_l2=1e-4)
    inp2 = attn_inputs(cfg, seed=62)
    out2, lse2, ref_out2, _ = _run_pair(cfg, inp2, want_lse=False, H_kv=H_kv)
    assert lse2 is None
    assert_close(out2, ref_out2, "factored call out")


def test_noalloc_matches_oracle():
    # One direct comparison with the float64 oracle (not only with the other
    # entry point), with an exact-range frozen head among factored ones.
    B, H, T, d = 2, 4, 256, 64
    cfg = AttnConfig("noalloc_o", B=B, H=H, T=T, d_h=d, dtype="bf16", static_heads=(1, 2))
    inp = attn_inputs(cfg, seed=71)
    inp["alpha"][2] = (0.45 * np.arange(T) - 40.0).astype(np.float32)
    out, lse, _, _ = _run_pair(cfg, inp)
    Q, K, V = (bf16_round(inp[n]) for n in ("Q", "K", "V"))
    ref_out, ref_lse = oracle.hybrid_attn_fwd(Q, K, V, inp["alpha"], inp["rho"],
                                              cfg.head_is_static)
    st = cfg.head_is_static.astype(bool)
    for cls, sel in (("static", st), ("dynamic", ~st)):
        assert_close(out[:, sel], ref_out[:, sel], f"oracle out[{cls}]")
        assert_close(lse[:, sel], ref_lse[:, sel], f"oracle lse[{cls}]", atol=1e-3, rel_l2=1e-4)


@pytest.mark.parametrize("n_static,T", [LIMIT_OK, LIMIT_OK2])
def test_noalloc_largest_fitting_shapes(n_static, T):
    # The largest scratch shapes run and agree with the workspace forward;
    # the frozen heads' rows are also spot-checked against the oracle.
    B, H, d = 1, n_static + 1, 64
    cfg = AttnConfig("noalloc_max", B=B, H=H, T=T, d_h=d, dtype="bf16",
                     static_heads=tuple(range(1, H)))
    inp = attn_inputs(cfg, seed=81)
    out, lse, ref_out, ref_lse = _run_pair(cfg, inp)
    assert_close(out, ref_out, "max shape out")
    assert_close(lse, ref_lse, "max shape lse", atol=1e-3, rel_l2=1e-4)
    rows = np.array([0, 1, 127, 128, T // 2 + 5, T - 1])
    for h in (1, H - 1):
        ro, rl = oracle.static_head_fwd_rows(inp["alpha"][h], inp["rho"][h],
                                             bf16_round(inp["V"][0, h]), rows)
        assert_close(out[0, h, rows], ro, f"max shape oracle out h{h}")
        assert_close(lse[0, h, rows], rl, f"max shape oracle lse h{h}", atol=1e-3, rel_l2=1e-4)


def test_noalloc_rejects_over_the_limit_before_launching():
    from dynamic_causal_attention_gb300 import _binding as B
    from dynamic_causal_attention_gb300 import api

    n_static, T = LIMIT_OVER
    H, d = n_static + 1, 64
    mask = np.zeros(H, dtype=np.uint8)
    mask[1:] = 1
    layer = api.HybridAttention(1, H, T, d, mask)
    v = torch.zeros((1, H, T, d), dtype=torch.bfloat16, device="cuda")
    q = torch.zeros_like(v)
    out = torch.zeros_like(v)
    ab = torch.zeros((H, T), dtype=torch.float32, device="cuda")
    st = _call_noalloc(B, layer, q, q, v, ab, ab, out, None)
    assert st == B.SAF_ERR_UNSUPPORTED, B.saf_status_string(st)
    assert B.saf_last_launch_count() == 0
    # and a regular call right after it still works and counts its launches
    mask2 = np.zeros(2, dtype=np.uint8)
    mask2[1] = 1
    small = api.HybridAttention(1, 2, 256, d, mask2)
    v2 = torch.randn((1, 2, 256, d), device="cuda").to(torch.bfloat16)
    ab2 = torch.zeros((2, 256), dtype=torch.float32, device="cuda")
    out2 = torch.empty_like(v2)
    st = _call_noalloc(B, small, v2, v2, v2, ab2, ab2, out2, None)
    assert st == B.SAF_OK, B.saf_status_string(st)
    assert B.saf_last_launch_count() == 2  # the frozen-head pre-pass and the forward
    torch.cuda.synchronize()
