"""The layer's C-ABI calls captured in a CUDA graph and replayed.

saf_hybrid_attn_fwd and saf_hybrid_attn_bwd, given a workspace, allocate
nothing and never synchronise with the host, so a training loop can capture
one step in a CUDA graph and replay it on the same buffers (the bench's
headline loop does).  Each replay must redo everything the step depends on:
the frozen heads' tables from the current alpha/rho, the status word, the
zeroed dQ accumulator.  Here a step is captured once; then new inputs are
copied into the captured buffers and the replay's results are compared with
an eager call on the same inputs (the forward bit for bit, the backward
within the run-to-run bounds of its fp32 reduce-adds) and with the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close, bf16_round, to_np
from dynamic_causal_attention_gb300.synthetic import AttnConfig, attn_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d_h", [64, 128])
def test_captured_step_replays_on_new_inputs(d_h):
    from dynamic_causal_attention_gb300 import api
    cfg = AttnConfig("graph", B=2, H=4, T=384, d_h=d_h, dtype="bf16", static_heads=(1,))
    first = attn_inputs(cfg, seed=101)
    dev = torch.device("cuda")
    buf = {n: torch.from_numpy(first[n]).to(dev, torch.bfloat16) for n in ("Q", "K", "V", "dO")}
    buf["alpha"] = torch.from_numpy(first["alpha"]).to(dev)
    buf["rho"] = torch.from_numpy(first["rho"]).to(dev)
    layer = api.HybridAttention(cfg.B, cfg.H, cfg.T, cfg.d_h, cfg.head_is_static,
                                want_param_grads=True)
    shp = (cfg.B, cfg.H, cfg.T, cfg.d_h)
    out = torch.empty(shp, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(shp[:3], dtype=torch.float32, device=dev)
    grads = tuple(torch.empty(shp, dtype=torch.bfloat16, device=dev) for _ in range(3)) + (
        torch.empty((cfg.H, cfg.T), device=dev), torch.empty((cfg.H, cfg.T), device=dev))

    def step():
        layer.forward(buf["Q"], buf["K"], buf["V"], buf["alpha"], buf["rho"], out=out, lse=lse)
        layer.backward(buf["Q"], buf["K"], buf["V"], out, lse, buf["dO"], buf["alpha"],
                       buf["rho"], want_param_grads=True, grads=grads)

    step()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step()
    torch.cuda.synchronize()

    # new inputs (a different frozen-head pattern too) into the captured buffers
    second = attn_inputs(cfg, seed=202)
    second["alpha"] = (second["alpha"] * 1.5).astype(np.float32)
    for n in ("Q", "K", "V", "dO"):
        buf[n].copy_(torch.from_numpy(second[n]).to(dev, torch.bfloat16))
    buf["alpha"].copy_(torch.from_numpy(second["alpha"]))
    buf["rho"].copy_(torch.from_numpy(second["rho"]))
    g.replay()
    torch.cuda.synchronize()
    st, site = layer.device_status()
    assert st == 0, site
    replayed = [to_np(out), to_np(lse)] + [to_np(t) for t in grads]

    step()                                        # eager, same inputs
    torch.cuda.synchronize()
    eager = [to_np(out), to_np(lse)] + [to_np(t) for t in grads]
    np.testing.assert_array_equal(replayed[0], eager[0])      # out
    np.testing.assert_array_equal(replayed[1], eager[1])      # lse
    np.testing.assert_array_equal(replayed[3], eager[3])      # dK
    np.testing.assert_array_equal(replayed[4], eager[4])      # dV
    dq_r, dq_e = replayed[2], eager[2]
    assert np.all(np.abs(dq_r - dq_e) <= 2.0 ** -7 * np.maximum(np.abs(dq_r), np.abs(dq_e))
                  + 1e-6 * np.abs(dq_e).max())

    # and against the oracle
    Q, K, V, dO = (bf16_round(second[n]) for n in ("Q", "K", "V", "dO"))
    ref_out, _ = oracle.hybrid_attn_fwd(Q, K, V, second["alpha"], second["rho"],
                                        cfg.head_is_static)
    assert_close(replayed[0], ref_out, "replayed out")
    rq, rk, rv, ra, rr = oracle.hybrid_attn_bwd(Q, K, V, second["alpha"], second["rho"],
                                                cfg.head_is_static, dO, True)
    dyn = ~np.asarray(cfg.head_is_static, bool)
    assert_close(replayed[2][:, dyn], rq[:, dyn], "replayed dQ")
    assert_close(replayed[4], rv, "replayed dV")
    st_ = np.asarray(cfg.head_is_static, bool)
    assert_close(replayed[5][st_], ra[st_], "replayed dalpha")
    assert_close(replayed[6][st_], rr[st_], "replayed drho")
