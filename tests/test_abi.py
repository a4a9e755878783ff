"""Host-side checks of the C ABI (no GPU needed).

The library must load on a machine without a GPU, export every entry point
that include/la.h declares, and reject bad arguments on the host before any
CUDA call (the header promises checks happen before any launch).
"""
import ctypes
import os
import re

import pytest

from weight_recurrence_gb300 import build as labuild
from weight_recurrence_gb300 import la

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "la.h")


@pytest.fixture(scope="module")
def lib():
    labuild.build()
    return la.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_]+)\s*\(", src)))


def test_header_declares_expected_calls():
    assert set(_declared()) == set(la.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings(lib):
    for st in range(6):
        assert la.status_string(st)
    assert la.status_string(la.LA_ERR_BOUNDS) != la.status_string(la.LA_ERR_TIMEOUT)
    assert la.status_string(la.LA_ERR_TIMEOUT) != la.status_string(la.LA_OK)
    assert la.la_version() >= 10000


def _shape(B=1, H=1, N=8, D=16, M=16, dt=la.LA_DTYPE_F32):
    return la.la_shape(B, H, N, D, M, dt)


FAKE = ctypes.c_void_p(0x10000)          # aligned, never dereferenced: checks fail first
MISALIGNED = ctypes.c_void_p(0x10008)


def test_workspace_query(lib):
    assert la.la_workspace_bytes(la.LA_OP_DECODE, _shape()) == 0
    assert la.la_workspace_bytes(la.LA_OP_CAUSAL, _shape()) >= 0
    assert la.la_workspace_bytes(la.LA_OP_NONCAUSAL, _shape(N=4096, D=64, M=64)) > 0
    with pytest.raises(la.LAError):
        la.la_workspace_bytes(la.LA_OP_CAUSAL, _shape(D=48))
    with pytest.raises(la.LAError):
        la.la_workspace_bytes(la.LA_OP_CAUSAL, _shape(), chunk=96)


@pytest.mark.parametrize("D,M", [(8, 16), (16, 24), (256, 64), (64, 0)])
def test_unsupported_dims(lib, D, M):
    st = lib.la_forward_causal(FAKE, FAKE, FAKE, FAKE, _shape(D=D, M=M), 0, None, None, None, 0, None)
    assert st == la.LA_ERR_UNSUPPORTED
    st = lib.la_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, _shape(D=D, M=M), None)
    assert st == la.LA_ERR_UNSUPPORTED


def test_invalid_arguments(lib):
    sh = _shape()
    # negative sizes / unknown dtype
    assert lib.la_forward_causal(FAKE, FAKE, FAKE, FAKE, _shape(N=-1), 0, None, None, None, 0, None) \
        == la.LA_ERR_INVALID_ARG
    assert lib.la_forward_noncausal(FAKE, FAKE, FAKE, FAKE, _shape(B=-2), None, 0, None) \
        == la.LA_ERR_INVALID_ARG
    assert lib.la_forward_causal(FAKE, FAKE, FAKE, FAKE, _shape(dt=7), 0, None, None, None, 0, None) \
        == la.LA_ERR_INVALID_ARG
    # null and misaligned pointers
    assert lib.la_forward_causal(None, FAKE, FAKE, FAKE, sh, 0, None, None, None, 0, None) \
        == la.LA_ERR_INVALID_ARG
    assert lib.la_forward_causal(FAKE, MISALIGNED, FAKE, FAKE, sh, 0, None, None, None, 0, None) \
        == la.LA_ERR_INVALID_ARG
    assert lib.la_decode_step(FAKE, FAKE, FAKE, FAKE, None, FAKE, sh, None) == la.LA_ERR_INVALID_ARG
    # exactly one of S, z given
    assert lib.la_forward_causal(FAKE, FAKE, FAKE, FAKE, sh, 0, FAKE, None, None, 0, None) \
        == la.LA_ERR_INVALID_ARG
    # unsupported chunk length
    assert lib.la_forward_causal(FAKE, FAKE, FAKE, FAKE, sh, 96, None, None, None, 0, None) \
        == la.LA_ERR_UNSUPPORTED
    # workspace too small for the non-causal reduction
    big = _shape(N=4096, D=64, M=64)
    assert lib.la_forward_noncausal(FAKE, FAKE, FAKE, ctypes.c_void_p(0x20000), big, FAKE, 16, None) \
        == la.LA_ERR_INVALID_ARG
    # output aliasing an input
    assert lib.la_forward_causal(FAKE, ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000), FAKE, sh, 0,
                                 None, None, None, 0, None) == la.LA_ERR_INVALID_ARG


def test_empty_problems_are_noops(lib):
    # nothing to compute -> OK without touching the (fake) buffers or any device
    assert lib.la_forward_causal(None, None, None, None, _shape(N=0), 0, None, None, None, 0, None) == la.LA_OK
    assert lib.la_forward_noncausal(None, None, None, None, _shape(B=0), None, 0, None) == la.LA_OK
    assert lib.la_decode_step(None, None, None, None, None, None, _shape(H=0), None) == la.LA_OK


def _addr(i):
    return ctypes.c_void_p(0x100000 * (i + 1))


def test_backward_argument_checks(lib):
    sh = _shape(N=64, D=16, M=16)
    q, k, v, g, dq, dk, dv = (_addr(i) for i in range(7))
    ws_c = la.la_workspace_bytes(la.LA_OP_CAUSAL_BWD, sh)
    ws_n = la.la_workspace_bytes(la.LA_OP_NONCAUSAL_BWD, sh)
    # g and e of every token, and two segment sums (one segment at N = 64)
    assert ws_c == 1 * 1 * 64 * (16 + 1) * 4 + 2 * (16 * 16 + 16) * 4
    assert ws_n > 0
    args = (q, k, v, g, dq, dk, dv, sh)
    # exactly one of each state pair given
    for pos in range(6):
        st = [None] * 6
        st[pos] = FAKE
        assert lib.la_backward_causal(*args, *st, _addr(9), ws_c, None) == la.LA_ERR_INVALID_ARG
    # workspace too small / missing
    assert lib.la_backward_causal(*args, None, None, None, None, None, None, _addr(9), ws_c - 4, None) \
        == la.LA_ERR_INVALID_ARG
    assert lib.la_backward_noncausal(*args, None, 0, None) == la.LA_ERR_INVALID_ARG
    # gradient aliasing an input, or another gradient
    assert lib.la_backward_causal(q, k, v, g, k, dk, dv, sh, None, None, None, None, None, None, _addr(9), ws_c,
                                  None) == la.LA_ERR_INVALID_ARG
    assert lib.la_backward_noncausal(q, k, v, g, dq, dq, dv, sh, _addr(9), ws_n, None) == la.LA_ERR_INVALID_ARG
    # misaligned input, unsupported width
    assert lib.la_backward_noncausal(MISALIGNED, k, v, g, dq, dk, dv, sh, _addr(9), ws_n, None) \
        == la.LA_ERR_INVALID_ARG
    assert lib.la_backward_causal(*args[:7], _shape(D=48), None, None, None, None, None, None, None, 0, None) \
        == la.LA_ERR_UNSUPPORTED
    # empty problems launch nothing
    assert lib.la_backward_noncausal(None, None, None, None, None, None, None, _shape(N=0), None, 0, None) \
        == la.LA_OK
    assert lib.la_backward_causal(None, None, None, None, None, None, None, _shape(B=0), None, None, None, None,
                                  None, None, None, 0, None) == la.LA_OK


def test_generation_argument_checks(lib):
    sh = _shape(B=2, N=64, D=16, M=16)
    q, k, v, o = (_addr(i) for i in range(4))
    # per-sequence lengths are required and 4-byte aligned
    assert lib.la_forward_causal_varlen(q, k, v, o, None, sh, None, None, None, 0, None) == la.LA_ERR_INVALID_ARG
    assert lib.la_forward_causal_varlen(q, k, v, o, ctypes.c_void_p(0x10002), sh, None, None, None, 0, None) \
        == la.LA_ERR_INVALID_ARG
    assert lib.la_forward_causal_varlen(q, k, v, o, _addr(5), sh, FAKE, None, None, 0, None) == la.LA_ERR_INVALID_ARG
    assert lib.la_forward_causal_varlen(None, None, None, None, None, _shape(N=0), None, None, None, 0, None) \
        == la.LA_OK
    # negative step count, misaligned step counts, missing state
    assert lib.la_decode_steps(q, k, v, o, _addr(5), _addr(6), None, -1, sh, None) == la.LA_ERR_INVALID_ARG
    assert lib.la_decode_steps(q, k, v, o, _addr(5), _addr(6), ctypes.c_void_p(0x10002), 4, sh, None) \
        == la.LA_ERR_INVALID_ARG
    assert lib.la_decode_steps(q, k, v, o, None, _addr(6), None, 4, sh, None) == la.LA_ERR_INVALID_ARG
    assert lib.la_decode_steps(None, None, None, None, None, None, None, 0, sh, None) == la.LA_OK
    assert lib.la_decode_steps(q, k, v, o, _addr(5), _addr(6), None, 4, _shape(D=24), None) == la.LA_ERR_UNSUPPORTED


def test_variant_feature_dims(lib):
    V = la.variant
    assert la.la_feature_dim(V("elu1"), 64) == 64
    assert la.la_feature_dim(V("dpfp", 1, "sum"), 64) == 128
    assert la.la_feature_dim(V("dpfp", 3, "none"), 64) == 384
    assert la.la_feature_dim(V("poly2", 1, "den"), 16) == 256
    assert la.la_feature_dim(V("dpfp", 0, "sum"), 64) == 0            # nu out of range
    assert la.la_feature_dim(la.la_variant(7, 1, 0, 0), 64) == 0       # unknown feature map


def test_variant_argument_checks(lib):
    V = la.variant
    sh = _shape(B=2, N=64, D=16, M=16)
    q, k, v, b, o, S, z = (_addr(i) for i in range(7))
    call = lib.la_forward_causal_variant
    # unsupported combinations
    assert call(q, k, v, None, o, sh, V("dpfp", 1, "den"), None, None, None) == la.LA_ERR_UNSUPPORTED
    assert call(q, k, v, None, o, sh, V("poly2", 1, "sum"), None, None, None) == la.LA_ERR_UNSUPPORTED
    assert call(q, k, v, b, o, sh, V("elu1", 1, "den", "delta"), S, z, None) == la.LA_ERR_UNSUPPORTED
    assert call(q, k, v, None, o, _shape(D=64), V("poly2", 1, "den"), None, None, None) \
        == la.LA_ERR_UNSUPPORTED                                      # F = 4096 > 512
    assert call(q, k, v, None, o, _shape(D=128), V("dpfp", 3, "sum"), None, None, None) \
        == la.LA_ERR_UNSUPPORTED                                      # F = 768 > 512
    # unknown enum values, nu out of range
    assert call(q, k, v, None, o, sh, la.la_variant(0, 1, 5, 0), None, None, None) == la.LA_ERR_INVALID_ARG
    assert call(q, k, v, None, o, sh, la.la_variant(0, 1, 0, 3), None, None, None) == la.LA_ERR_INVALID_ARG
    assert call(q, k, v, None, o, sh, V("dpfp", 40, "sum"), None, None, None) == la.LA_ERR_INVALID_ARG
    # delta rule needs beta; z only with the denominator; S and z together there
    assert call(q, k, v, None, o, sh, V("elu1", 1, "sum", "delta"), None, None, None) == la.LA_ERR_INVALID_ARG
    assert call(q, k, v, None, o, sh, V("elu1", 1, "sum"), S, z, None) == la.LA_ERR_INVALID_ARG
    assert call(q, k, v, None, o, sh, V("elu1", 1, "den"), S, None, None) == la.LA_ERR_INVALID_ARG
    assert call(q, k, v, None, o, sh, V("elu1", 1, "den"), None, z, None) == la.LA_ERR_INVALID_ARG
    # misaligned, aliasing, empty
    assert call(MISALIGNED, k, v, None, o, sh, V(), None, None, None) == la.LA_ERR_INVALID_ARG
    assert call(q, k, v, None, q, sh, V(), None, None, None) == la.LA_ERR_INVALID_ARG
    assert call(None, None, None, None, None, _shape(N=0), V("dpfp", 2, "none"), None, None, None) == la.LA_OK
    # non-causal: sum update only; workspace
    nc = lib.la_forward_noncausal_variant
    need = la.lib().la_variant_workspace_bytes(la.LA_OP_NONCAUSAL, sh, V("dpfp", 1, "sum"))
    assert need == 2 * 2 * (32 * 16 + 32) * 4                      # 2 heads, 2 key splits, F = 2 * 16
    assert nc(q, k, v, o, sh, V("elu1", 1, "sum", "delta"), _addr(9), 1 << 20, None) == la.LA_ERR_UNSUPPORTED
    assert nc(q, k, v, o, sh, V("dpfp", 1, "sum"), _addr(9), need - 4, None) == la.LA_ERR_INVALID_ARG
    assert nc(None, None, None, None, _shape(B=0), V(), None, 0, None) == la.LA_OK
    # decode: the state is required
    dec = lib.la_decode_step_variant
    assert dec(q, k, v, None, o, None, None, sh, V("elu1", 1, "sum"), None) == la.LA_ERR_INVALID_ARG
    assert dec(q, k, v, None, o, S, None, sh, V("elu1", 1, "sum", "delta"), None) == la.LA_ERR_INVALID_ARG
    assert dec(None, None, None, None, None, None, None, _shape(B=0), V(), None) == la.LA_OK


def test_checked_build_exports_the_same_abi(lib):
    """The bounds-checked twin builds from the same sources, exports every
    declared entry point and says which build it is."""
    path = labuild.build(checked=True)
    assert path == la.LIB_CHECKED_PATH
    checked = la._load(path)
    for name in _declared():
        assert ctypes.cast(getattr(checked, name), ctypes.c_void_p).value, name
    assert checked.la_checked_build() == 1
    assert lib.la_checked_build() == 0
    # selecting a build routes the module's calls, and back
    try:
        assert la.select_library(True) is checked and la.la_checked_build()
        la.la_debug_inject_bounds(False)   # host-side flag only: no device work
    finally:
        la.select_library(False)
    assert not la.la_checked_build()


@pytest.mark.parametrize("B,H,N,D,M", [(1, 16, 65536, 128, 128), (16, 8, 3072, 128, 128), (1, 1, 4097, 128, 64),
                                       (64, 4, 700, 64, 128), (300, 1, 128, 128, 128)])
def test_segmented_backward_workspace(lib, B, H, N, D, M):
    """bf16 causal backward at D, M in {64, 128} (not 64/64) takes the segmented
    route: its workspace holds g (bf16) and e of every token, and two fp32
    [S | z] slots per segment for the most segments any device picks (up to
    192 SMs: one CTA per SM, at least one segment per head, at most one per
    128-row chunk), each part on a 256-byte boundary."""
    def up(b):
        return (b + 255) // 256 * 256
    sh = _shape(B=B, H=H, N=N, D=D, M=M, dt=la.LA_DTYPE_BF16)
    BH, nch = B * H, (N + 127) // 128
    nseg = max(1, min(nch, 192 // BH))
    L = (nch + nseg - 1) // nseg
    nseg = (nch + L - 1) // L
    seg = 2 * up(BH * nseg * (D * M + D) * 4) + up(BH * N * M * 2) + BH * N * 4
    # the CUDA-core route's need is the floor (the two share the call's workspace)
    assert la.la_workspace_bytes(la.LA_OP_CAUSAL_BWD, sh) >= seg
    # fp32 at the same sizes runs on CUDA cores: g and e per token, two segment sums
    fp = la.la_workspace_bytes(la.LA_OP_CAUSAL_BWD, _shape(B=B, H=H, N=N, D=D, M=M))
    assert fp >= BH * N * (M + 1) * 4
