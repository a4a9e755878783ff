"""fp64 CPU oracle for kernelised linear attention, phi(x) = elu(x) + 1.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``, never by the product package.  It
shares no code with the CUDA library.

Two independent forms, both written from "Transformers are RNNs" (read in
its Chinese translation):

* ``recurrence`` (C, ``la_oracle.c``): sec. 3.3 eqs. (10)-(12) and sec. 3.4
  eqs. (16)-(20) walked token by token in fp64 loops; also sec. 3.2 eq. (5)
  for the non-causal form.  This is also the timed CPU baseline.
* ``definition`` (numpy, ``definition.py``): sec. 3.1 eq. (3) with
  sim(q, k) = phi(q)^T phi(k) (sec. 3.2 eq. (4)) and the causal mask of
  sec. 3.3 eq. (8), as a dense quadratic form.
* ``causal_backward`` / ``noncausal_backward`` (C): gradients by the chain
  rule through eqs. (10)-(12) (forward sweep for dQ, reverse cumulative sums
  for dK, dV - the constant-memory scheme sec. 3.3.1 describes, whose own
  equations (13)-(15) the page does not print).

Parity status: pinned (see tests/test_oracle.py) by the hand-derived fixtures
under tests/golden/, closed forms, invariants and planted-mistake checks; the
backward (tests/test_oracle_backward.py) by central finite differences and by
autograd of the definition form, closed forms and planted-mistake checks.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .definition import definition_causal, definition_noncausal, definition_rows, phi_np  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liblaoracle.so")
_SRC = os.path.join(_HERE, "la_oracle.c")
_lib = None


def build(force: bool = False) -> str:
    """Compile la_oracle.c with gcc (-O2 -fopenmp); returns the .so path."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_SO)
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        L = ctypes.c_long
        dp = ctypes.c_void_p
        lib.lao_phi.restype = ctypes.c_double
        lib.lao_phi.argtypes = [ctypes.c_double]
        lib.lao_max_threads.restype = ctypes.c_int
        lib.lao_causal_mut.restype = ctypes.c_int
        lib.lao_causal_mut.argtypes = [f32p, f32p, f32p, L, L, L, L, dp, dp, dp, dp, dp,
                                       ctypes.c_int, ctypes.c_int]
        lib.lao_noncausal_mut.restype = ctypes.c_int
        lib.lao_noncausal_mut.argtypes = [f32p, f32p, f32p, L, L, L, L, dp, dp, dp,
                                          ctypes.c_int, ctypes.c_int]
        lib.lao_decode.restype = ctypes.c_int
        lib.lao_decode.argtypes = [f32p, f32p, f32p, L, L, L, dp, dp, dp, ctypes.c_int]
        lib.lao_causal_backward_mut.restype = ctypes.c_int
        lib.lao_causal_backward_mut.argtypes = [f32p, f32p, f32p, f32p, L, L, L, L, dp, dp, dp, dp,
                                                dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int]
        lib.lao_noncausal_backward_mut.restype = ctypes.c_int
        lib.lao_noncausal_backward_mut.argtypes = [f32p, f32p, f32p, f32p, L, L, L, L, dp, dp, dp,
                                                   ctypes.c_int, ctypes.c_int]
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(x) -> np.ndarray:
    """Widen to a contiguous fp32 numpy array (exact for bf16 and fp32 data)."""
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def phi(x: float) -> float:
    """phi(x) = elu(x) + 1 evaluated by the C oracle in fp64 (sec. 3.2.1 eq. (7))."""
    return _load().lao_phi(float(x))


def max_threads() -> int:
    return int(_load().lao_max_threads())


def causal(q, k, v, S0=None, z0=None, want_out=True, nthreads=0, mutant=0):
    """Causal recurrence, eqs. (10)-(12) / (16)-(20).

    q, k: [..., N, D]; v: [..., N, M] (any leading batch/head dims).
    Returns (out [..., N, M] fp64 or None, S [..., D, M] fp64, z [..., D] fp64).
    """
    q, k, v = _f32(q), _f32(k), _f32(v)
    lead = q.shape[:-2]
    N, D = q.shape[-2], q.shape[-1]
    M = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (N, M), np.float64) if want_out else None
    S = np.empty(lead + (D, M), np.float64)
    z = np.empty(lead + (D,), np.float64)
    S0a = None if S0 is None else np.ascontiguousarray(np.asarray(S0, np.float64).reshape(lead + (D, M)))
    z0a = None if z0 is None else np.ascontiguousarray(np.asarray(z0, np.float64).reshape(lead + (D,)))
    rc = _load().lao_causal_mut(q.reshape(-1), k.reshape(-1), v.reshape(-1), BH, N, D, M,
                                _ptr(S0a), _ptr(z0a), _ptr(out), _ptr(S), _ptr(z),
                                int(nthreads), int(mutant))
    if rc != 0:
        raise ValueError("oracle: bad shape")
    return out, S, z


def noncausal(q, k, v, nthreads=0, mutant=0):
    """Non-causal form, eq. (5).  Returns (out, KV = sum phi(K)V^T, ksum = sum phi(K))."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    lead = q.shape[:-2]
    N, D = q.shape[-2], q.shape[-1]
    M = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (N, M), np.float64)
    kv = np.empty(lead + (D, M), np.float64)
    ks = np.empty(lead + (D,), np.float64)
    rc = _load().lao_noncausal_mut(q.reshape(-1), k.reshape(-1), v.reshape(-1), BH, N, D, M,
                                   _ptr(out), _ptr(kv), _ptr(ks), int(nthreads), int(mutant))
    if rc != 0:
        raise ValueError("oracle: bad shape")
    return out, kv, ks


def decode_step(q, k, v, S, z, nthreads=0):
    """One recurrent step, eqs. (18)-(20).  S [..., D, M] and z [..., D] (fp64) are
    updated in place; returns y [..., M] fp64."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    D, M = q.shape[-1], v.shape[-1]
    lead = q.shape[:-1]
    BH = int(np.prod(lead)) if lead else 1
    assert S.dtype == np.float64 and S.flags.c_contiguous and z.dtype == np.float64
    y = np.empty(lead + (M,), np.float64)
    rc = _load().lao_decode(q.reshape(-1), k.reshape(-1), v.reshape(-1), BH, D, M,
                            _ptr(S), _ptr(z), _ptr(y), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: bad shape")
    return y


def _f64_or_none(x, shape):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x.detach().cpu().double().numpy() if hasattr(x, "detach") else x,
                                           np.float64).reshape(shape))


def causal_backward(q, k, v, G, S0=None, z0=None, dSN=None, dzN=None, nthreads=0, mutant=0):
    """Gradients through the causal form, eqs. (9)-(12), given G = dL/dV'.

    q, k: [..., N, D]; v, G: [..., N, M].  S0/z0: carried-in state (or None);
    dSN/dzN: gradient reaching the final state (or None).  Returns
    (dq, dk, dv, dS0, dz0), all fp64; dS0/dz0 are dL/dS_0, dL/dZ_0."""
    q, k, v, G = _f32(q), _f32(k), _f32(v), _f32(G)
    lead = q.shape[:-2]
    N, D = q.shape[-2], q.shape[-1]
    M = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    dq = np.empty(lead + (N, D), np.float64)
    dk = np.empty(lead + (N, D), np.float64)
    dv = np.empty(lead + (N, M), np.float64)
    dS0 = np.empty(lead + (D, M), np.float64)
    dz0 = np.empty(lead + (D,), np.float64)
    S0a, z0a = _f64_or_none(S0, lead + (D, M)), _f64_or_none(z0, lead + (D,))
    dSa, dza = _f64_or_none(dSN, lead + (D, M)), _f64_or_none(dzN, lead + (D,))
    rc = _load().lao_causal_backward_mut(q.reshape(-1), k.reshape(-1), v.reshape(-1), G.reshape(-1),
                                         BH, N, D, M, _ptr(S0a), _ptr(z0a), _ptr(dSa), _ptr(dza),
                                         _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dS0), _ptr(dz0),
                                         int(nthreads), int(mutant))
    if rc != 0:
        raise ValueError("oracle: bad shape")
    return dq, dk, dv, dS0, dz0


def noncausal_backward(q, k, v, G, nthreads=0, mutant=0):
    """Gradients through the non-causal form, eq. (5), given G = dL/dV'.
    Returns (dq, dk, dv) in fp64."""
    q, k, v, G = _f32(q), _f32(k), _f32(v), _f32(G)
    lead = q.shape[:-2]
    N, D = q.shape[-2], q.shape[-1]
    M = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    dq = np.empty(lead + (N, D), np.float64)
    dk = np.empty(lead + (N, D), np.float64)
    dv = np.empty(lead + (N, M), np.float64)
    rc = _load().lao_noncausal_backward_mut(q.reshape(-1), k.reshape(-1), v.reshape(-1), G.reshape(-1),
                                            BH, N, D, M, _ptr(dq), _ptr(dk), _ptr(dv),
                                            int(nthreads), int(mutant))
    if rc != 0:
        raise ValueError("oracle: bad shape")
    return dq, dk, dv


# Planted-mistake identifiers of la_oracle.c (test use only).
MUTANTS = {
    "relu": 1, "no_z_update": 2, "read_before_update": 3, "transpose_S": 4,
    "phi_sign": 5, "shifted_v": 6, "den_uses_k": 7,
    # backward
    "bwd_no_e": 11, "bwd_dphi_is_phi": 12, "bwd_excl_diag": 13, "bwd_dv_uses_q": 14,
}
