"""Torch-facing entry points of libsaf (device memory and streams only).

These wrappers allocate outputs and the workspace with torch, pass raw
device addresses and the current CUDA stream to the C ABI, and raise on any
non-OK status.  All arithmetic runs in libsaf's kernels.
"""

from __future__ import annotations

import numpy as np
import torch

from . import _binding as B

__all__ = ["HybridAttention", "Calibration", "fit_compact", "num_select", "SafError"]

SafError = B.SafError


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device=None):
    return torch.cuda.current_stream(device).cuda_stream


def _check(st, where):
    if st != B.SAF_OK:
        raise B.SafError(st, where)


class HybridAttention:
    """One hybrid causal attention layer of shape (B, H, T, d_h).

    ``head_is_static`` marks the frozen heads (host booleans, length H).
    ``dtype`` is torch.bfloat16 or torch.float32 (fp32 I/O is computed in
    bf16 inside the library).  ``H_kv`` < H groups the K/V heads: query head
    h reads K/V head h // (H // H_kv), and K, V, dK, dV are [B, H_kv, T, d_h].
    """

    def __init__(self, B_: int, H: int, T: int, d_h: int, head_is_static,
                 dtype=torch.bfloat16, device="cuda", want_param_grads=False, H_kv=None):
        self.shape = (B_, H, T, d_h)
        self.H_kv = H if H_kv is None else H_kv
        self.dtype = dtype
        self.device = torch.device(device)
        code = B.SAF_BF16 if dtype == torch.bfloat16 else B.SAF_F32
        self.dims = B._dims(B_, H, T, d_h, code, self.H_kv)
        self.head_is_static = bytes(np.asarray(head_is_static, dtype=np.uint8).tolist())
        assert len(self.head_is_static) == H
        self.ws_bytes = B.saf_hybrid_attn_workspace_size(self.dims, int(want_param_grads))
        if self.ws_bytes == 0:
            raise B.SafError(B.SAF_ERR_UNSUPPORTED, "saf_hybrid_attn_workspace_size")
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=self.device)

    def forward(self, q, k, v, alpha, rho, out=None, lse=None):
        B_, H, T, d = self.shape
        if out is None:
            out = torch.empty((B_, H, T, d), dtype=self.dtype, device=self.device)
        if lse is None:
            lse = torch.empty((B_, H, T), dtype=torch.float32, device=self.device)
        st = B.saf_hybrid_attn_fwd(self.dims, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(rho),
                                   self.head_is_static, _ptr(out), _ptr(lse),
                                   _ptr(self.workspace), self.ws_bytes, _stream(self.device))
        _check(st, "saf_hybrid_attn_fwd")
        return out, lse

    def backward(self, q, k, v, out, lse, dout, alpha, rho, want_param_grads=False,
                 grads=None):
        B_, H, T, d = self.shape
        if grads is None:
            mk = lambda h: torch.empty((B_, h, T, d), dtype=self.dtype, device=self.device)
            dq, dk, dv = mk(H), mk(self.H_kv), mk(self.H_kv)
            da = dr = None
            if want_param_grads:
                da = torch.empty((H, T), dtype=torch.float32, device=self.device)
                dr = torch.empty((H, T), dtype=torch.float32, device=self.device)
        else:
            dq, dk, dv, da, dr = grads
        st = B.saf_hybrid_attn_bwd(self.dims, _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                   _ptr(dout), _ptr(alpha), _ptr(rho), self.head_is_static,
                                   _ptr(dq), _ptr(dk), _ptr(dv), _ptr(da), _ptr(dr),
                                   _ptr(self.workspace), self.ws_bytes, _stream(self.device))
        _check(st, "saf_hybrid_attn_bwd")
        return dq, dk, dv, da, dr

    def device_status(self):
        return B.saf_get_device_status(_ptr(self.workspace), 0, _stream(self.device))


class Calibration:
    """Streaming calibration state for ``num_heads`` heads of length T."""

    def __init__(self, num_heads: int, T: int, device="cuda", track_kl=False):
        self.device = torch.device(device)
        with torch.cuda.device(self.device):
            st, self.handle = B.saf_calib_create_ex(
                num_heads, T, B.SAF_CALIB_TRACK_KL if track_kl else 0)
        _check(st, "saf_calib_create_ex")
        self.num_heads, self.T = num_heads, T

    def accumulate(self, A, head_begin=0):
        n, hc = A.shape[0], A.shape[1]
        st = B.saf_calib_accumulate(self.handle, _ptr(A), n, head_begin, hc, _stream(self.device))
        _check(st, "saf_calib_accumulate")

    def finalize(self, k, want_mean=True):
        A_hat = None
        if want_mean:
            A_hat = torch.empty((self.num_heads, self.T, self.T), dtype=torch.float32,
                                device=self.device)
        s_var = torch.empty(self.num_heads, dtype=torch.float32, device=self.device)
        sel = torch.empty(max(k, 1), dtype=torch.int32, device=self.device)
        st = B.saf_calib_finalize(self.handle, k, _ptr(A_hat), _ptr(s_var), _ptr(sel),
                                  _stream(self.device))
        _check(st, "saf_calib_finalize")
        return A_hat, s_var, sel[:k]

    def finalize_kl(self, k):
        """Forward-KL selector: (s_kl [num_heads], the k lowest-scoring heads)."""
        s_kl = torch.empty(self.num_heads, dtype=torch.float32, device=self.device)
        sel = torch.empty(max(k, 1), dtype=torch.int32, device=self.device)
        st = B.saf_calib_finalize_kl(self.handle, k, _ptr(s_kl), _ptr(sel), _stream(self.device))
        _check(st, "saf_calib_finalize_kl")
        return s_kl, sel[:k]

    def finalize_sharp(self):
        """Sharp-mean pattern [num_heads, T, T] of a handle fed logits: the
        causal softmax of each row of the logits' mean."""
        out = torch.empty((self.num_heads, self.T, self.T), dtype=torch.float32,
                          device=self.device)
        st = B.saf_calib_finalize_sharp(self.handle, _ptr(out), _stream(self.device))
        _check(st, "saf_calib_finalize_sharp")
        return out

    def reset(self):
        _check(B.saf_calib_reset(self.handle), "saf_calib_reset")

    def close(self):
        if self.handle is not None:
            B.saf_calib_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def fit_compact(A_hat, candidates, k, kl_max=0.2, steps=400, lr=1e-2):
    """Fit alpha/rho to A_hat [num_heads, T, T] for each candidate head (device
    int32, priority order) and select the first k that pass the KL gate.
    Returns (alpha [n, T], rho [n, T], kl [n], selected [n_selected])."""
    num_heads, T, _ = A_hat.shape
    n = candidates.numel()
    dev = A_hat.device
    alpha = torch.empty((n, T), dtype=torch.float32, device=dev)
    rho = torch.empty((n, T), dtype=torch.float32, device=dev)
    kl = torch.empty(n, dtype=torch.float32, device=dev)
    sel = torch.empty(max(k, 1), dtype=torch.int32, device=dev)
    n_sel = torch.zeros(1, dtype=torch.int32, device=dev)
    st = B.saf_fit_compact(_ptr(A_hat), num_heads, T, _ptr(candidates), n, k, kl_max, steps, lr,
                           _ptr(alpha), _ptr(rho), _ptr(kl), _ptr(sel), _ptr(n_sel),
                           _stream(dev))
    _check(st, "saf_fit_compact")
    return alpha, rho, kl, sel[: int(n_sel.item())]


def num_select(r: float, num_heads: int) -> int:
    return B.saf_calib_num_select(r, num_heads)
