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
* ``variant_*`` (C, ``la_variants.c``): the same recurrence with the other
  feature maps (DPFP-nu of "Linear Transformers Are Secretly Fast Weight
  Programmers", the degree-2 polynomial map of sec. 3.2.1), sum-normalised
  features without a denominator, and the delta update rule with a per-token
  beta; ``definition_variant`` (numpy) is their quadratic form (sum update).
* ``causal_backward`` / ``noncausal_backward`` (C): gradients by the chain
  rule through eqs. (10)-(12) (forward sweep for dQ, reverse cumulative sums
  for dK, dV - the constant-memory scheme sec. 3.3.1 describes, whose own
  equations (13)-(15) the page does not print).

Parity status: pinned (see tests/test_oracle.py) by the hand-derived fixtures
under tests/golden/, closed forms, invariants and planted-mistake checks; the
backward (tests/test_oracle_backward.py) by central finite differences and by
autograd of the definition form, closed forms and planted-mistake checks; the
variants (tests/test_oracle_variants.py) by hand-derived features, the
polynomial kernel's closed form, the definition form, an independent chunked
(UT-transform) evaluation of the delta rule, closed forms of the delta rule
with one-hot keys, and planted-mistake checks.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .definition import (definition_causal, definition_noncausal, definition_rows,  # noqa: F401
                         definition_variant, features_np, phi_np)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liblaoracle.so")
_SRCS = [os.path.join(_HERE, "la_oracle.c"), os.path.join(_HERE, "la_variants.c")]
_lib = None


def build(force: bool = False) -> str:
    """Compile la_oracle.c and la_variants.c with gcc (-O2 -fopenmp); returns the .so path."""
    newest = max(os.path.getmtime(s) for s in _SRCS)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < newest:
        tmp = _SO + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp] + _SRCS + ["-lm"])
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
        I = ctypes.c_int
        lib.lav_feature_dim.restype = L
        lib.lav_feature_dim.argtypes = [I, L, I]
        lib.lav_features.restype = I
        lib.lav_features.argtypes = [f32p, L, L, I, I, I, dp]
        lib.lav_causal_mut.restype = I
        lib.lav_causal_mut.argtypes = [f32p, f32p, f32p, dp, L, L, L, L, I, I, I, I,
                                       dp, dp, dp, dp, dp, I, I]
        lib.lav_noncausal.restype = I
        lib.lav_noncausal.argtypes = [f32p, f32p, f32p, L, L, L, L, I, I, I, dp, I]
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


# Variant identifiers of la_variants.c (feature map, read-out normalisation, update rule).
FEATURE_MAPS = {"elu1": 0, "dpfp": 1, "poly2": 2}
NORMS = {"den": 0, "sum": 1, "none": 2}
UPDATES = {"sum": 0, "delta": 1}
VARIANT_MUTANTS = {"dpfp_pos_only": 21, "poly_upper": 22, "sumnorm_k_only": 23,
                   "delta_after": 24, "delta_sign": 25, "delta_beta_v": 26}


def feature_dim(fm: str, D: int, nu: int = 1) -> int:
    """F, the width of phi(x) for x in R^D (0 if the variant is invalid)."""
    return int(_load().lav_feature_dim(FEATURE_MAPS[fm], int(D), int(nu)))


def features(x, fm: str, nu: int = 1, sumnorm: bool = False) -> np.ndarray:
    """phi of every row of x [..., D] -> [..., F] in fp64 (C loops)."""
    x = _f32(x)
    D = x.shape[-1]
    F = feature_dim(fm, D, nu)
    R = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    out = np.empty(x.shape[:-1] + (F,), np.float64)
    rc = _load().lav_features(x.reshape(-1), R, D, FEATURE_MAPS[fm], int(nu), int(bool(sumnorm)), _ptr(out))
    if rc != 0:
        raise ValueError("oracle: bad feature map")
    return out


def variant_causal(q, k, v, fm="elu1", nu=1, norm="den", update="sum", beta=None,
                   S0=None, z0=None, want_out=True, nthreads=0, mutant=0):
    """Causal recurrence of a variant (la_variants.c).

    q, k: [..., N, D]; v: [..., N, M]; beta: [..., N] (delta update).
    Returns (out [..., N, M] or None, S [..., F, M], z [..., F]), fp64."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    lead = q.shape[:-2]
    N, D = q.shape[-2], q.shape[-1]
    M = v.shape[-1]
    F = feature_dim(fm, D, nu)
    BH = int(np.prod(lead)) if lead else 1
    b = None if beta is None else _f32(beta).reshape(-1)
    out = np.empty(lead + (N, M), np.float64) if want_out else None
    S = np.empty(lead + (F, M), np.float64)
    z = np.empty(lead + (F,), np.float64)
    S0a, z0a = _f64_or_none(S0, lead + (F, M)), _f64_or_none(z0, lead + (F,))
    rc = _load().lav_causal_mut(q.reshape(-1), k.reshape(-1), v.reshape(-1), _ptr(b), BH, N, D, M,
                                FEATURE_MAPS[fm], int(nu), NORMS[norm], UPDATES[update],
                                _ptr(S0a), _ptr(z0a), _ptr(out), _ptr(S), _ptr(z),
                                int(nthreads), int(mutant))
    if rc != 0:
        raise ValueError("oracle: bad variant or shape")
    return out, S, z


def variant_noncausal(q, k, v, fm="elu1", nu=1, norm="den", nthreads=0):
    """Non-causal form of a variant (sum update).  Returns out [..., N, M] fp64."""
    q, k, v = _f32(q), _f32(k), _f32(v)
    lead = q.shape[:-2]
    N, D = q.shape[-2], q.shape[-1]
    M = v.shape[-1]
    BH = int(np.prod(lead)) if lead else 1
    out = np.empty(lead + (N, M), np.float64)
    rc = _load().lav_noncausal(q.reshape(-1), k.reshape(-1), v.reshape(-1), BH, N, D, M,
                               FEATURE_MAPS[fm], int(nu), NORMS[norm], _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle: bad variant or shape")
    return out
