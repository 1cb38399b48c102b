"""The workspace-free forward entry point, checked against the regular one.

saf_hybrid_attn_fwd_noalloc is for callers that cannot allocate device memory
while they run the layer, such as an engine plugin that is handed only its
input and output buffers because the engine planned all memory in advance.
Its scratch is one fixed device array inside the library, shared by every call
and keeping the last call's contents, so the test makes two calls in a row on
different inputs and compares each with saf_hybrid_attn_fwd (which uses a
caller-provided workspace) on the same inputs.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes when run alone.
"""

import numpy as np
import pytest
import torch

from helpers import assert_close, to_dev, to_np
from dynamic_causal_attention_gb300.synthetic import AttnConfig, attn_inputs

pytestmark = pytest.mark.gpu


def test_noalloc_forward_matches_workspace_forward_twice():
    from dynamic_causal_attention_gb300 import _binding as B
    from dynamic_causal_attention_gb300 import api

    cfg = AttnConfig("noalloc", B=2, H=6, T=512, d_h=64, dtype="bf16", static_heads=(1, 4))
    stream = torch.cuda.current_stream().cuda_stream
    for call, seed in enumerate((51, 52)):
        inp = attn_inputs(cfg, seed=seed)
        if call == 1:
            # a different pattern on the second call: stale tables would show
            inp["alpha"] *= 2.0
            inp["rho"] = (inp["rho"] * 0.5).astype(np.float32)
        q, k, v = (to_dev(inp[n], torch.bfloat16) for n in ("Q", "K", "V"))
        alpha = to_dev(inp["alpha"], torch.float32)
        rho = to_dev(inp["rho"], torch.float32)
        layer = api.HybridAttention(cfg.B, cfg.H, cfg.T, cfg.d_h, cfg.head_is_static)
        ref_out, ref_lse = layer.forward(q, k, v, alpha, rho)
        out = torch.full_like(ref_out, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        st = B.saf_hybrid_attn_fwd_noalloc(layer.dims, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                           alpha.data_ptr(), rho.data_ptr(), layer.head_is_static,
                                           out.data_ptr(), lse.data_ptr(), stream)
        assert st == B.SAF_OK, B.saf_status_string(st)
        torch.cuda.synchronize()
        assert_close(to_np(out), to_np(ref_out), f"call {call} out")
        assert_close(to_np(lse), to_np(ref_lse), f"call {call} lse", atol=1e-3, rel_l2=1e-4)
