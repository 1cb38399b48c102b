"""Host-side checks of the C ABI: the library builds, loads, exports every
symbol that include/saf.h declares, and rejects bad arguments before any
CUDA work (so these run without a GPU)."""

import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "saf.h")


@pytest.fixture(scope="module")
def binding():
    from dynamic_causal_attention_gb300 import _build
    if not os.path.exists(_build.LIB):
        _build.build()
    from dynamic_causal_attention_gb300 import _binding
    return _binding


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SAF_API\s+[\w\s\*]+?\b(saf_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("saf_hybrid_attn_fwd", "saf_hybrid_attn_bwd", "saf_calib_accumulate",
              "saf_calib_finalize", "saf_hybrid_attn_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(binding):
    lib = ctypes.CDLL(binding.LIB_PATH)
    for name in declared_symbols():
        assert hasattr(lib, name), f"libsaf.so does not export {name}"
    assert sorted(binding.EXPORTED) == declared_symbols()


def test_status_strings(binding):
    for code, name in [(0, "SAF_OK"), (1, "SAF_ERR_INVALID_ARG"), (2, "SAF_ERR_UNSUPPORTED"),
                       (3, "SAF_ERR_CUDA"), (4, "SAF_ERR_STATE"), (5, "SAF_ERR_TIMEOUT")]:
        assert binding.saf_status_string(code) == name


def test_num_select_half_to_even(binding):
    import oracle
    for r, n in [(0.25, 144), (0.125, 12), (0.25, 10), (0.5, 12), (0.0, 12), (1.0, 12),
                 (0.375, 4), (0.1, 15)]:
        assert binding.saf_calib_num_select(r, n) == oracle.num_select(r, n)


def test_workspace_size_and_unsupported_shapes(binding):
    d = binding._dims
    assert binding.saf_hybrid_attn_workspace_size(d(8, 12, 4096, 64, 0), 0) > 0
    assert binding.saf_hybrid_attn_workspace_size(d(1, 4, 128, 32, 1), 1) > 0
    # a length that is not a multiple of 128 runs on padded copies: the
    # workspace holds them (and more than the padded length's own workspace)
    ws_ragged = binding.saf_hybrid_attn_workspace_size(d(1, 4, 100, 32, 0), 0)
    assert ws_ragged > binding.saf_hybrid_attn_workspace_size(d(1, 4, 128, 32, 0), 0)
    assert binding.saf_hybrid_attn_workspace_size(d(1, 4, 16385, 32, 0), 0) == 0   # T
    assert binding.saf_hybrid_attn_workspace_size(d(1, 4, 128, 48, 0), 0) == 0   # d_h
    assert binding.saf_hybrid_attn_workspace_size(d(1, 300, 128, 64, 0), 0) == 0  # H
    assert binding.saf_hybrid_attn_workspace_size(d(0, 4, 128, 64, 0), 0) == 0   # empty
    assert binding.saf_hybrid_attn_workspace_size(d(-1, 4, 128, 64, 0), 0) == 0  # B
    # grouped K/V: H_kv must divide H; the grouped layout needs the extra dV sum
    ws_mha = binding.saf_hybrid_attn_workspace_size(d(2, 8, 256, 64, 0), 0)
    ws_gqa = binding.saf_hybrid_attn_workspace_size(d(2, 8, 256, 64, 0, 2), 0)
    assert ws_mha == binding.saf_hybrid_attn_workspace_size(d(2, 8, 256, 64, 0, 8), 0)
    assert ws_gqa > 0 and ws_gqa != ws_mha
    assert binding.saf_hybrid_attn_workspace_size(d(2, 8, 256, 64, 0, 3), 0) == 0
    assert binding.saf_hybrid_attn_workspace_size(d(2, 8, 256, 64, 0, -1), 0) == 0


def test_invalid_arguments_rejected_before_launch(binding):
    d = binding._dims
    hs = bytes([1, 0, 0, 0])
    # unsupported head dim -> UNSUPPORTED, nothing touched
    st = binding.saf_hybrid_attn_fwd(d(1, 4, 128, 48, 0), 16, 16, 16, 16, 16, hs, 16, 16,
                                     256, 1 << 30, None)
    assert st == binding.SAF_ERR_UNSUPPORTED
    # null V
    st = binding.saf_hybrid_attn_fwd(d(1, 4, 128, 64, 0), 16, 16, None, 16, 16, hs, 16, 16,
                                     256, 1 << 30, None)
    assert st == binding.SAF_ERR_INVALID_ARG
    # misaligned pointer
    st = binding.saf_hybrid_attn_fwd(d(1, 4, 128, 64, 0), 16, 16, 24, 16, 16, hs, 16, 16,
                                     256, 1 << 30, None)
    assert st == binding.SAF_ERR_INVALID_ARG
    # workspace too small
    st = binding.saf_hybrid_attn_fwd(d(1, 4, 128, 64, 0), 16, 16, 16, 16, 16, hs, 16, 16,
                                     256, 16, None)
    assert st == binding.SAF_ERR_INVALID_ARG
    # bwd: dalpha without drho
    st = binding.saf_hybrid_attn_bwd(d(1, 4, 128, 64, 0), 16, 16, 16, 16, 16, 16, 16, 16, hs,
                                     16, 16, 16, 16, None, 256, 1 << 30, None)
    assert st == binding.SAF_ERR_INVALID_ARG
    # bwd: missing lse
    st = binding.saf_hybrid_attn_bwd(d(1, 4, 128, 64, 0), 16, 16, 16, 16, None, 16, 16, 16, hs,
                                     16, 16, 16, None, None, 256, 1 << 30, None)
    assert st == binding.SAF_ERR_INVALID_ARG
    # static heads need alpha/rho
    st = binding.saf_hybrid_attn_fwd(d(1, 4, 128, 64, 0), 16, 16, 16, None, 16, hs, 16, 16,
                                     256, 1 << 30, None)
    assert st == binding.SAF_ERR_INVALID_ARG


def test_calib_argument_checks(binding):
    st, h = binding.saf_calib_create(0, 64)
    assert st == binding.SAF_ERR_INVALID_ARG and not h
    st, h = binding.saf_calib_create(4, 66)
    assert st == binding.SAF_ERR_INVALID_ARG
    assert binding.saf_calib_accumulate(None, 16, 1, 0, 1, None) == binding.SAF_ERR_INVALID_ARG
    assert binding.saf_calib_finalize(None, 0, None, 16, None, None) == binding.SAF_ERR_INVALID_ARG
    assert binding.saf_calib_destroy(None) == binding.SAF_OK


def test_noalloc_forward_rejects_what_its_scratch_cannot_hold(binding):
    d = binding._dims
    # 64 frozen heads at T = 16384 need ~16.8 MB of tables: beyond the 4 MiB array
    hs = bytes([1] * 64)
    st = binding.saf_hybrid_attn_fwd_noalloc(d(1, 64, 16384, 64, 0), 16, 16, 16, 16, 16, hs,
                                             16, 16, None)
    assert st == binding.SAF_ERR_UNSUPPORTED
    # fp32 I/O and lengths that are not a multiple of 128 would need staging buffers
    st = binding.saf_hybrid_attn_fwd_noalloc(d(1, 4, 128, 32, 1), 16, 16, 16, 16, 16,
                                             bytes([1, 0, 0, 0]), 16, 16, None)
    assert st == binding.SAF_ERR_UNSUPPORTED
    st = binding.saf_hybrid_attn_fwd_noalloc(d(1, 4, 200, 32, 0), 16, 16, 16, 16, 16,
                                             bytes([1, 0, 0, 0]), 16, 16, None)
    assert st == binding.SAF_ERR_UNSUPPORTED
    st = binding.saf_hybrid_attn_fwd_noalloc(d(1, 4, 128, 32, 0), 16, 16, None, 16, 16,
                                             bytes([1, 0, 0, 0]), 16, 16, None)
    assert st == binding.SAF_ERR_INVALID_ARG


def test_empty_layers_are_no_ops(binding):
    # B, H or T zero: SAF_OK at once, no pointer read (all None here), nothing
    # launched.  Invalid fields are still rejected.
    d = binding._dims
    for dims in (d(0, 4, 128, 64, 0), d(2, 0, 128, 64, 0), d(2, 4, 0, 64, 0)):
        st = binding.saf_hybrid_attn_fwd(dims, None, None, None, None, None, b"", None, None,
                                         None, 0, None)
        assert st == binding.SAF_OK, binding.saf_status_string(st)
        assert binding.saf_last_launch_count() == 0
        st = binding.saf_hybrid_attn_bwd(dims, None, None, None, None, None, None, None, None,
                                         b"", None, None, None, None, None, None, 0, None)
        assert st == binding.SAF_OK, binding.saf_status_string(st)
        assert binding.saf_last_launch_count() == 0
        st = binding.saf_hybrid_attn_fwd_noalloc(dims, None, None, None, None, None, b"",
                                                 None, None, None)
        assert st == binding.SAF_OK, binding.saf_status_string(st)
    bad = d(0, 4, 128, 48, 0)   # d_h is still checked
    assert binding.saf_hybrid_attn_fwd(bad, None, None, None, None, None, b"", None, None,
                                       None, 0, None) == binding.SAF_ERR_UNSUPPORTED
    neg = d(-2, 4, 128, 64, 0)
    assert binding.saf_hybrid_attn_fwd(neg, None, None, None, None, None, b"", None, None,
                                       None, 0, None) == binding.SAF_ERR_INVALID_ARG
