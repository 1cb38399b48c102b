"""ctypes binding of libsaf's C ABI (include/saf.h): argument marshalling only.

Every function here has the name and argument order of the C entry point it
wraps.  Device buffers are passed as integer addresses (or None for NULL),
``head_is_static`` as a host byte sequence, streams as integer
``cudaStream_t`` handles.  There is no fallback: importing this module fails
if the compiled library is missing.
"""

from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsaf.so")

SAF_OK = 0
SAF_ERR_INVALID_ARG = 1
SAF_ERR_UNSUPPORTED = 2
SAF_ERR_CUDA = 3
SAF_ERR_STATE = 4
SAF_ERR_TIMEOUT = 5

SAF_BF16 = 0
SAF_F32 = 1

SAF_CALIB_TRACK_KL = 1

EXPORTED = (
    "saf_hybrid_attn_workspace_size",
    "saf_hybrid_attn_fwd",
    "saf_hybrid_attn_bwd",
    "saf_hybrid_attn_fwd_noalloc",
    "saf_calib_create",
    "saf_calib_create_ex",
    "saf_calib_accumulate",
    "saf_calib_num_select",
    "saf_calib_finalize",
    "saf_calib_finalize_kl",
    "saf_calib_finalize_sharp",
    "saf_fit_compact",
    "saf_calib_reset",
    "saf_calib_destroy",
    "saf_get_device_status",
    "saf_status_string",
    "saf_last_launch_count",
    "saf_trace_enable",
    "saf_trace_count",
    "saf_trace_get",
    "saf_debug_forward_hold",
)


class saf_attn_dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
                ("d_h", ctypes.c_int), ("dtype", ctypes.c_int), ("H_kv", ctypes.c_int)]


class SafError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {saf_status_string(status)} ({status})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libsaf.so is not built ({LIB_PATH}); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    return ctypes.CDLL(LIB_PATH)


_lib = _load()
_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t

_lib.saf_hybrid_attn_workspace_size.argtypes = [ctypes.POINTER(saf_attn_dims), _i]
_lib.saf_hybrid_attn_workspace_size.restype = _sz
_lib.saf_hybrid_attn_fwd.argtypes = [ctypes.POINTER(saf_attn_dims), _vp, _vp, _vp, _vp, _vp,
                                     ctypes.c_char_p, _vp, _vp, _vp, _sz, _vp]
_lib.saf_hybrid_attn_fwd.restype = _i
_lib.saf_hybrid_attn_bwd.argtypes = [ctypes.POINTER(saf_attn_dims), _vp, _vp, _vp, _vp, _vp,
                                     _vp, _vp, _vp, ctypes.c_char_p, _vp, _vp, _vp, _vp, _vp,
                                     _vp, _sz, _vp]
_lib.saf_hybrid_attn_bwd.restype = _i
_lib.saf_hybrid_attn_fwd_noalloc.argtypes = [ctypes.POINTER(saf_attn_dims), _vp, _vp, _vp, _vp,
                                             _vp, ctypes.c_char_p, _vp, _vp, _vp]
_lib.saf_hybrid_attn_fwd_noalloc.restype = _i
_lib.saf_calib_create.argtypes = [ctypes.POINTER(_vp), _i, _i]
_lib.saf_calib_create.restype = _i
_lib.saf_calib_create_ex.argtypes = [ctypes.POINTER(_vp), _i, _i, ctypes.c_uint]
_lib.saf_calib_create_ex.restype = _i
_lib.saf_calib_finalize_kl.argtypes = [_vp, _i, _vp, _vp, _vp]
_lib.saf_calib_finalize_kl.restype = _i
_lib.saf_calib_finalize_sharp.argtypes = [_vp, _vp, _vp]
_lib.saf_calib_finalize_sharp.restype = _i
_lib.saf_calib_accumulate.argtypes = [_vp, _vp, _i, _i, _i, _vp]
_lib.saf_calib_accumulate.restype = _i
_lib.saf_calib_num_select.argtypes = [ctypes.c_double, _i]
_lib.saf_calib_num_select.restype = _i
_lib.saf_calib_finalize.argtypes = [_vp, _i, _vp, _vp, _vp, _vp]
_lib.saf_calib_finalize.restype = _i
_lib.saf_fit_compact.argtypes = [_vp, _i, _i, _vp, _i, _i, ctypes.c_float, _i, ctypes.c_float,
                                 _vp, _vp, _vp, _vp, _vp, _vp]
_lib.saf_fit_compact.restype = _i
_lib.saf_calib_reset.argtypes = [_vp]
_lib.saf_calib_reset.restype = _i
_lib.saf_calib_destroy.argtypes = [_vp]
_lib.saf_calib_destroy.restype = _i
_lib.saf_get_device_status.argtypes = [_vp, _i, ctypes.POINTER(_i), _vp]
_lib.saf_get_device_status.restype = _i
_lib.saf_status_string.argtypes = [_i]
_lib.saf_status_string.restype = ctypes.c_char_p
_lib.saf_last_launch_count.argtypes = []
_lib.saf_last_launch_count.restype = _i
_lib.saf_trace_enable.argtypes = [_i]
_lib.saf_trace_enable.restype = _i
_lib.saf_trace_count.argtypes = []
_lib.saf_trace_count.restype = _i
_lib.saf_trace_get.argtypes = [_i, ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float)]
_lib.saf_trace_get.restype = _i
_lib.saf_debug_forward_hold.argtypes = [_i]
_lib.saf_debug_forward_hold.restype = _i


def lib():
    return _lib


def _dims(B, H, T, d_h, dtype, H_kv=0):
    return saf_attn_dims(int(B), int(H), int(T), int(d_h), int(dtype), int(H_kv))


def saf_status_string(status: int) -> str:
    return _lib.saf_status_string(int(status)).decode()


def saf_last_launch_count() -> int:
    return _lib.saf_last_launch_count()


def saf_trace_enable(enable: int) -> int:
    return _lib.saf_trace_enable(int(enable))


def saf_trace_count() -> int:
    return _lib.saf_trace_count()


def saf_debug_forward_hold(hold: int) -> int:
    return _lib.saf_debug_forward_hold(int(hold))


def saf_trace_get(index: int):
    name = ctypes.c_char_p()
    ms = ctypes.c_float()
    st = _lib.saf_trace_get(int(index), ctypes.byref(name), ctypes.byref(ms))
    return st, (name.value.decode() if name.value else None), ms.value


def saf_hybrid_attn_workspace_size(dims: saf_attn_dims, want_param_grads: int) -> int:
    return _lib.saf_hybrid_attn_workspace_size(ctypes.byref(dims), int(want_param_grads))


def saf_hybrid_attn_fwd(dims, Q, K, V, alpha, rho, head_is_static: bytes, out, lse,
                        workspace, ws_bytes, stream) -> int:
    return _lib.saf_hybrid_attn_fwd(ctypes.byref(dims), Q, K, V, alpha, rho,
                                    bytes(head_is_static), out, lse, workspace,
                                    int(ws_bytes), stream)


def saf_hybrid_attn_bwd(dims, Q, K, V, out, lse, dout, alpha, rho, head_is_static: bytes,
                        dQ, dK, dV, dalpha, drho, workspace, ws_bytes, stream) -> int:
    return _lib.saf_hybrid_attn_bwd(ctypes.byref(dims), Q, K, V, out, lse, dout, alpha, rho,
                                    bytes(head_is_static), dQ, dK, dV, dalpha, drho,
                                    workspace, int(ws_bytes), stream)


def saf_hybrid_attn_fwd_noalloc(dims, Q, K, V, alpha, rho, head_is_static: bytes, out, lse,
                                stream) -> int:
    return _lib.saf_hybrid_attn_fwd_noalloc(ctypes.byref(dims), Q, K, V, alpha, rho,
                                            bytes(head_is_static), out, lse, stream)


def saf_calib_create(num_heads: int, T: int):
    h = _vp()
    st = _lib.saf_calib_create(ctypes.byref(h), int(num_heads), int(T))
    return st, h.value


def saf_calib_create_ex(num_heads: int, T: int, flags: int):
    h = _vp()
    st = _lib.saf_calib_create_ex(ctypes.byref(h), int(num_heads), int(T), int(flags))
    return st, h.value


def saf_calib_finalize_kl(handle, k, s_kl, selected, stream) -> int:
    return _lib.saf_calib_finalize_kl(handle, int(k), s_kl, selected, stream)


def saf_calib_finalize_sharp(handle, pattern, stream) -> int:
    return _lib.saf_calib_finalize_sharp(handle, pattern, stream)


def saf_calib_accumulate(handle, A, n, head_begin, head_count, stream) -> int:
    return _lib.saf_calib_accumulate(handle, A, int(n), int(head_begin), int(head_count), stream)


def saf_calib_num_select(r: float, num_heads: int) -> int:
    return _lib.saf_calib_num_select(float(r), int(num_heads))


def saf_calib_finalize(handle, k, A_hat, s_var, selected, stream) -> int:
    return _lib.saf_calib_finalize(handle, int(k), A_hat, s_var, selected, stream)


def saf_fit_compact(A_hat, num_heads, T, candidates, n_candidates, k, kl_max, steps, lr,
                    alpha, rho, kl, selected, n_selected, stream) -> int:
    return _lib.saf_fit_compact(A_hat, int(num_heads), int(T), candidates, int(n_candidates),
                                int(k), float(kl_max), int(steps), float(lr), alpha, rho, kl,
                                selected, n_selected, stream)


def saf_calib_reset(handle) -> int:
    return _lib.saf_calib_reset(handle)


def saf_calib_destroy(handle) -> int:
    return _lib.saf_calib_destroy(handle)


def saf_get_device_status(workspace_or_handle, is_calib_handle, stream):
    site = _i(0)
    st = _lib.saf_get_device_status(workspace_or_handle, int(is_calib_handle),
                                    ctypes.byref(site), stream)
    return st, site.value
