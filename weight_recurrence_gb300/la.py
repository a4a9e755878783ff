"""ctypes binding of liblinattn.so (argument marshalling only).

Every function here has the name of the C entry point it calls (see
``include/la.h``) and takes torch tensors for the device buffers; torch
provides device memory and the current CUDA stream, nothing else.  All work
runs in the library's kernels.  If the library is missing the first call
raises: there is no fallback.

Two builds of the library exist: liblinattn.so (the product) and
liblinattn_checked.so, the same kernels compiled with in-kernel bounds checks
that record LA_ERR_BOUNDS in the error word instead of making an access out
of range.  The environment variable LA_CHECKED=1 (read at the first load) or
select_library(checked=True) makes every call below go to the checked build.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "liblinattn.so")
LIB_CHECKED_PATH = os.path.join(_PKG, "lib", "liblinattn_checked.so")

LA_OK, LA_ERR_INVALID_ARG, LA_ERR_UNSUPPORTED, LA_ERR_CUDA, LA_ERR_TIMEOUT, LA_ERR_BOUNDS = range(6)
LA_DTYPE_F32, LA_DTYPE_BF16 = 0, 1
LA_OP_NONCAUSAL, LA_OP_CAUSAL, LA_OP_DECODE, LA_OP_NONCAUSAL_BWD, LA_OP_CAUSAL_BWD = 0, 1, 2, 3, 4

EXPORTED = ("la_workspace_bytes", "la_forward_noncausal", "la_forward_causal", "la_decode_step",
            "la_get_last_error", "la_status_string", "la_version", "la_launch_count",
            "la_debug_inject_timeout", "la_forward_noncausal_noalloc", "la_backward_causal",
            "la_backward_noncausal", "la_forward_causal_varlen", "la_decode_steps",
            "la_feature_dim", "la_variant_workspace_bytes", "la_forward_causal_variant",
            "la_forward_noncausal_variant", "la_decode_step_variant", "la_checked_build",
            "la_debug_inject_bounds")

LA_FM = {"elu1": 0, "dpfp": 1, "poly2": 2}
LA_NORM = {"den": 0, "sum": 1, "none": 2}
LA_UPDATE = {"sum": 0, "delta": 1}


class LAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


class la_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int),
                ("D", ctypes.c_int), ("M", ctypes.c_int), ("dtype", ctypes.c_int)]


class la_variant(ctypes.Structure):
    _fields_ = [("feature_map", ctypes.c_int), ("nu", ctypes.c_int), ("norm", ctypes.c_int),
                ("update", ctypes.c_int)]


def variant(fm: str = "elu1", nu: int = 1, norm: str = "den", update: str = "sum") -> la_variant:
    """la_variant from names: fm in {"elu1", "dpfp", "poly2"}, norm in {"den",
    "sum", "none"}, update in {"sum", "delta"}."""
    return la_variant(LA_FM[fm], int(nu), LA_NORM[norm], LA_UPDATE[update])


_lib = None
_loaded = {}


def select_library(checked: bool) -> ctypes.CDLL:
    """Routes the calls of this module to the checked build (True) or to the
    product build (False); returns the library now in use."""
    global _lib
    _lib = _load(LIB_CHECKED_PATH if checked else LIB_PATH)
    return _lib


def lib() -> ctypes.CDLL:
    """The library in use (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = _load(LIB_CHECKED_PATH if os.environ.get("LA_CHECKED", "0") not in ("", "0") else LIB_PATH)
    return _lib


def _load(path: str) -> ctypes.CDLL:
    L = _loaded.get(path)
    if L is None:
        if not os.path.exists(path):
            flag = " --checked" if path == LIB_CHECKED_PATH else ""
            raise RuntimeError("%s is not built; run `python -m weight_recurrence_gb300.build%s`"
                               % (path, flag))
        L = ctypes.CDLL(path)
        vp, sz, i = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        L.la_workspace_bytes.restype = sz
        L.la_workspace_bytes.argtypes = [i, la_shape, i]
        L.la_forward_noncausal.restype = i
        L.la_forward_noncausal.argtypes = [vp, vp, vp, vp, la_shape, vp, sz, vp]
        L.la_forward_causal.restype = i
        L.la_forward_causal.argtypes = [vp, vp, vp, vp, la_shape, i, vp, vp, vp, sz, vp]
        L.la_decode_step.restype = i
        L.la_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, la_shape, vp]
        L.la_get_last_error.restype = i
        L.la_get_last_error.argtypes = [vp]
        L.la_status_string.restype = ctypes.c_char_p
        L.la_status_string.argtypes = [i]
        L.la_version.restype = i
        L.la_launch_count.restype = ctypes.c_ulonglong
        L.la_forward_noncausal_noalloc.restype = i
        L.la_forward_noncausal_noalloc.argtypes = [vp, vp, vp, vp, la_shape, vp]
        L.la_debug_inject_timeout.restype = None
        L.la_debug_inject_timeout.argtypes = [i, i]
        L.la_backward_causal.restype = i
        L.la_backward_causal.argtypes = [vp, vp, vp, vp, vp, vp, vp, la_shape, vp, vp, vp, vp, vp, vp, vp, sz, vp]
        L.la_forward_causal_varlen.restype = i
        L.la_forward_causal_varlen.argtypes = [vp, vp, vp, vp, vp, la_shape, vp, vp, vp, sz, vp]
        L.la_decode_steps.restype = i
        L.la_decode_steps.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, la_shape, vp]
        L.la_backward_noncausal.restype = i
        L.la_backward_noncausal.argtypes = [vp, vp, vp, vp, vp, vp, vp, la_shape, vp, sz, vp]
        L.la_feature_dim.restype = i
        L.la_feature_dim.argtypes = [la_variant, i]
        L.la_variant_workspace_bytes.restype = sz
        L.la_variant_workspace_bytes.argtypes = [i, la_shape, la_variant]
        L.la_forward_causal_variant.restype = i
        L.la_forward_causal_variant.argtypes = [vp, vp, vp, vp, vp, la_shape, la_variant, vp, vp, vp]
        L.la_forward_noncausal_variant.restype = i
        L.la_forward_noncausal_variant.argtypes = [vp, vp, vp, vp, la_shape, la_variant, vp, sz, vp]
        L.la_decode_step_variant.restype = i
        L.la_decode_step_variant.argtypes = [vp, vp, vp, vp, vp, vp, vp, la_shape, la_variant, vp]
        L.la_checked_build.restype = i
        L.la_checked_build.argtypes = []
        L.la_debug_inject_bounds.restype = None
        L.la_debug_inject_bounds.argtypes = [i]
        _loaded[path] = L
    return L


def status_string(st: int) -> str:
    return lib().la_status_string(int(st)).decode()


def _dtype_code(t: torch.dtype) -> int:
    if t == torch.float32:
        return LA_DTYPE_F32
    if t == torch.bfloat16:
        return LA_DTYPE_BF16
    raise TypeError("unsupported dtype %s (float32 or bfloat16)" % t)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _stream(stream, device):
    return ctypes.c_void_p(_stream_ptr(stream, device))


def _check(st: int, where: str):
    if st != LA_OK:
        raise LAError(st, where)


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def shape_of(q: torch.Tensor, v: torch.Tensor) -> la_shape:
    B, H, N, D = q.shape
    return la_shape(B, H, N, D, v.shape[-1], _dtype_code(q.dtype))


_SIZE_MAX = ctypes.c_size_t(-1).value
_ws_bytes_cache = {}


def la_workspace_bytes(op: int, shape: la_shape, chunk: int = 0) -> int:
    key = (int(op), shape.B, shape.H, shape.N, shape.D, shape.M, shape.dtype, int(chunk))
    n = _ws_bytes_cache.get(key)
    if n is None:
        n = lib().la_workspace_bytes(int(op), shape, int(chunk))
        if n == _SIZE_MAX:
            raise LAError(LA_ERR_INVALID_ARG, "la_workspace_bytes")
        _ws_bytes_cache[key] = n = int(n)
    return n


_ws_cache = {}


def _workspace(nbytes: int, device, stream_ptr: int) -> torch.Tensor | None:
    if nbytes == 0:
        return None
    key = (device.index, stream_ptr)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def la_forward_noncausal(q, k, v, out=None, stream=None):
    """V' = phi(Q)(phi(K)^T V) / phi(Q) sum phi(K) for q, k [B,H,N,D], v [B,H,N,M]."""
    _contig(q, k, v)
    s = shape_of(q, v)
    if out is None:
        out = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _contig(out)
    need = la_workspace_bytes(LA_OP_NONCAUSAL, s, 0)
    sp = _stream_ptr(stream, q.device)
    ws = _workspace(need, q.device, sp)
    st = lib().la_forward_noncausal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), s, _ptr(ws), need, ctypes.c_void_p(sp))
    _check(st, "la_forward_noncausal")
    return out


def la_forward_noncausal_noalloc(q, k, v, out=None, stream=None):
    """As la_forward_noncausal, but the library uses its own fixed 8 MiB device
    scratch array instead of a workspace (for callers that cannot allocate;
    overlapping calls race on that array)."""
    _contig(q, k, v)
    s = shape_of(q, v)
    if out is None:
        out = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _contig(out)
    st = lib().la_forward_noncausal_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), s, _stream(stream, q.device))
    _check(st, "la_forward_noncausal_noalloc")
    return out


def la_forward_causal(q, k, v, out=None, chunk=0, S=None, z=None, want_out=True, stream=None):
    """Causal form (sums over j <= i).  S [B,H,D,M] / z [B,H,D] fp32, if given,
    hold the carried-in state and receive the state after the last token."""
    _contig(q, k, v, S, z)
    s = shape_of(q, v)
    if out is None and want_out:
        out = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _contig(out)
    need = la_workspace_bytes(LA_OP_CAUSAL, s, chunk)
    sp = _stream_ptr(stream, q.device)
    ws = _workspace(need, q.device, sp)
    st = lib().la_forward_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(out), s, int(chunk), _ptr(S), _ptr(z),
                                 _ptr(ws), need, ctypes.c_void_p(sp))
    _check(st, "la_forward_causal")
    return out


def la_decode_step(q, k, v, S, z, y=None, stream=None):
    """One recurrent step for q, k [B,H,D], v [B,H,M]; S, z fp32 updated in place."""
    _contig(q, k, v, S, z)
    B, H, D = q.shape
    M = v.shape[-1]
    if y is None:
        y = torch.empty((B, H, M), dtype=q.dtype, device=q.device)
    _contig(y)
    s = la_shape(B, H, 1, D, M, _dtype_code(q.dtype))
    st = lib().la_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(S), _ptr(z), s,
                              _stream(stream, q.device))
    _check(st, "la_decode_step")
    return y


def la_forward_causal_varlen(q, k, v, lens, out=None, S=None, z=None, want_out=True, stream=None):
    """Causal form for a batch of sequences of lengths lens [B] (int32, on the
    device); rows past a sequence's length are ignored (their output rows are
    unspecified).  S, z as in la_forward_causal, per sequence."""
    _contig(q, k, v, S, z, lens)
    if lens.dtype != torch.int32:
        raise ValueError("lens must be int32")
    s = shape_of(q, v)
    if out is None and want_out:
        out = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _contig(out)
    need = la_workspace_bytes(LA_OP_CAUSAL, s, 0)
    sp = _stream_ptr(stream, q.device)
    ws = _workspace(need, q.device, sp)
    st = lib().la_forward_causal_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lens), s, _ptr(S), _ptr(z),
                                        _ptr(ws), need, ctypes.c_void_p(sp))
    _check(st, "la_forward_causal_varlen")
    return out


def la_decode_steps(q, k, v, S, z, y=None, steps=None, stream=None):
    """T recurrent steps in one launch: q, k [T,B,H,D], v [T,B,H,M]; S, z fp32
    updated in place; steps: optional int32 [B] per-sequence step counts."""
    _contig(q, k, v, S, z, steps)
    T, B, H, D = q.shape
    M = v.shape[-1]
    if y is None:
        y = torch.empty((T, B, H, M), dtype=q.dtype, device=q.device)
    _contig(y)
    if steps is not None and steps.dtype != torch.int32:
        raise ValueError("steps must be int32")
    s = la_shape(B, H, 1, D, M, _dtype_code(q.dtype))
    st = lib().la_decode_steps(_ptr(q), _ptr(k), _ptr(v), _ptr(y), _ptr(S), _ptr(z), _ptr(steps), int(T), s,
                               _stream(stream, q.device))
    _check(st, "la_decode_steps")
    return y


def la_backward_causal(q, k, v, dout, dq=None, dk=None, dv=None, S0=None, z0=None, dSN=None, dzN=None,
                       dS0=None, dz0=None, stream=None):
    """Gradients dq, dk, dv of the causal form given dout = dL/dV'.  S0/z0: the
    state the forward started from; dSN/dzN: gradient reaching its final
    state; dS0/dz0 (fp32, written): gradient of the starting state."""
    _contig(q, k, v, dout, S0, z0, dSN, dzN, dS0, dz0)
    s = shape_of(q, v)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _contig(dq, dk, dv)
    need = la_workspace_bytes(LA_OP_CAUSAL_BWD, s, 0)
    sp = _stream_ptr(stream, q.device)
    ws = _workspace(need, q.device, sp)
    st = lib().la_backward_causal(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), s,
                                  _ptr(S0), _ptr(z0), _ptr(dSN), _ptr(dzN), _ptr(dS0), _ptr(dz0),
                                  _ptr(ws), need, ctypes.c_void_p(sp))
    _check(st, "la_backward_causal")
    return dq, dk, dv


def la_backward_noncausal(q, k, v, dout, dq=None, dk=None, dv=None, stream=None):
    """Gradients dq, dk, dv of the non-causal form given dout = dL/dV'."""
    _contig(q, k, v, dout)
    s = shape_of(q, v)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _contig(dq, dk, dv)
    need = la_workspace_bytes(LA_OP_NONCAUSAL_BWD, s, 0)
    sp = _stream_ptr(stream, q.device)
    ws = _workspace(need, q.device, sp)
    st = lib().la_backward_noncausal(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), s,
                                     _ptr(ws), need, ctypes.c_void_p(sp))
    _check(st, "la_backward_noncausal")
    return dq, dk, dv


def la_feature_dim(var: la_variant, D: int) -> int:
    """Width F of phi(x) for x in R^D under the variant (0 if invalid)."""
    return int(lib().la_feature_dim(var, int(D)))


def la_forward_causal_variant(q, k, v, var: la_variant, beta=None, out=None, S=None, z=None, want_out=True,
                              stream=None):
    """Causal form of a variant: q, k [B,H,N,D], v [B,H,N,M], beta [B,H,N]
    (delta rule).  S [B,H,F,M] (and z [B,H,F] with the denominator) fp32, if
    given, hold the starting state and receive the final one."""
    _contig(q, k, v, beta, S, z)
    s = shape_of(q, v)
    if out is None and want_out:
        out = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _contig(out)
    st = lib().la_forward_causal_variant(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(out), s, var, _ptr(S),
                                         _ptr(z), _stream(stream, q.device))
    _check(st, "la_forward_causal_variant")
    return out


def la_forward_noncausal_variant(q, k, v, var: la_variant, out=None, stream=None):
    """Non-causal form of a variant (sum update)."""
    _contig(q, k, v)
    s = shape_of(q, v)
    if out is None:
        out = torch.empty(q.shape[:-1] + (v.shape[-1],), dtype=q.dtype, device=q.device)
    _contig(out)
    need = lib().la_variant_workspace_bytes(LA_OP_NONCAUSAL, s, var)
    if need == _SIZE_MAX:
        raise LAError(LA_ERR_UNSUPPORTED, "la_variant_workspace_bytes")
    sp = _stream_ptr(stream, q.device)
    ws = _workspace(int(need), q.device, sp)
    st = lib().la_forward_noncausal_variant(_ptr(q), _ptr(k), _ptr(v), _ptr(out), s, var, _ptr(ws), int(need),
                                            ctypes.c_void_p(sp))
    _check(st, "la_forward_noncausal_variant")
    return out


def la_decode_step_variant(q, k, v, S, var: la_variant, z=None, beta=None, y=None, stream=None):
    """One recurrent step of a variant: q, k [B,H,D], v [B,H,M], beta [B,H];
    S [B,H,F,M] (and z [B,H,F] with the denominator) updated in place."""
    _contig(q, k, v, S, z, beta)
    B, H, D = q.shape
    M = v.shape[-1]
    if y is None:
        y = torch.empty((B, H, M), dtype=q.dtype, device=q.device)
    _contig(y)
    s = la_shape(B, H, 1, D, M, _dtype_code(q.dtype))
    st = lib().la_decode_step_variant(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(y), _ptr(S), _ptr(z), s, var,
                                      _stream(stream, q.device))
    _check(st, "la_decode_step_variant")
    return y


def la_get_last_error(stream=None, device=None) -> int:
    """Synchronises the stream and returns (and clears) the device error word."""
    dev = device if device is not None else torch.cuda.current_device()
    return int(lib().la_get_last_error(_stream(stream, dev)))


def la_debug_inject_timeout(enable: bool, limit_us: int = 1000):
    lib().la_debug_inject_timeout(1 if enable else 0, int(limit_us))


def la_checked_build() -> bool:
    """True when the library in use is the bounds-checked build."""
    return bool(lib().la_checked_build())


def la_debug_inject_bounds(enable: bool):
    """Checked build only (a no-op otherwise): while enabled, the kernels that
    read a carried-in state or a workspace slot offset that index past its
    buffer, so that their check records LA_ERR_BOUNDS and skips the access."""
    lib().la_debug_inject_bounds(1 if enable else 0)


def la_version() -> int:
    return int(lib().la_version())


def la_launch_count() -> int:
    """Kernels launched through the library by this process so far."""
    return int(lib().la_launch_count())
