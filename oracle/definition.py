"""Definition form of kernelised attention, fp64 numpy (test infrastructure only).

Written from "Transformers are RNNs" (read in its Chinese translation):

* sec. 3.1 eq. (3): V'_i = sum_j sim(Q_i, K_j) V_j / sum_j sim(Q_i, K_j);
* sec. 3.2 eq. (4): sim(q, k) = phi(q)^T phi(k), phi applied row-wise;
* sec. 3.2.1 eq. (7): phi(x) = elu(x) + 1 (alpha = 1);
* sec. 3.3 eq. (8): the causal form sums over j <= i only.

This is the O(N^2) quadratic form the linear method avoids.  The matrix of
similarities is formed explicitly with one matmul; there is no regrouping.
"""
from __future__ import annotations

import numpy as np


def phi_np(x: np.ndarray) -> np.ndarray:
    """elu(x) + 1 in fp64: x + 1 for x > 0, exp(x) for x <= 0."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x > 0.0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _as64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().to("cpu").float().numpy()
    return np.asarray(a, dtype=np.float64)


def definition_noncausal(q, k, v) -> np.ndarray:
    """eq. (3)/(4) over all j.  q, k: [..., N, D]; v: [..., N, M]."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    w = phi_np(q) @ np.swapaxes(phi_np(k), -1, -2)          # sim(Q_i, K_j), [..., N, N]
    return (w @ v) / w.sum(axis=-1, keepdims=True)


def definition_causal(q, k, v) -> np.ndarray:
    """eq. (8) with the similarity of eq. (4): sums over j <= i."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    N = q.shape[-2]
    w = phi_np(q) @ np.swapaxes(phi_np(k), -1, -2)
    w = w * np.tril(np.ones((N, N)))                           # keep j <= i
    return (w @ v) / w.sum(axis=-1, keepdims=True)


def definition_rows(q, k, v, rows, causal: bool, prefix_state=None) -> np.ndarray:
    """eq. (3)/(8) for selected query rows only, for long sequences.

    q, k: [N, D], v: [N, M] of ONE head; rows: 1-D int array of query indices.
    Row i costs O(i * D) (causal) so sampled rows of a 64k sequence are cheap.
    ``prefix_state`` = (S0, z0) adds the contribution of tokens before this
    sequence (the state carried in): V'_i = (phi(q)^T S0 + sum ...) / (phi(q)^T z0 + sum ...).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    rows = np.asarray(rows, dtype=np.int64)
    fq = phi_np(q[rows])                                        # [R, D]
    out = np.empty((rows.size, v.shape[-1]), np.float64)
    for r, i in enumerate(rows):
        hi = i + 1 if causal else q.shape[0]
        w = phi_np(k[:hi]) @ fq[r]                               # [hi]
        num = w @ v[:hi]
        den = w.sum()
        if prefix_state is not None:
            S0, z0 = prefix_state
            num = num + fq[r] @ np.asarray(S0, np.float64)
            den = den + fq[r] @ np.asarray(z0, np.float64)
        out[r] = num / den
    return out


def features_np(x, fm: str, nu: int = 1, sumnorm: bool = False) -> np.ndarray:
    """The variants' feature maps in vectorised numpy fp64, [..., D] -> [..., F].

    * "elu1": eq. (7) of "Transformers are RNNs".
    * "dpfp": DPFP-nu of "Linear Transformers Are Secretly Fast Weight
      Programmers": r = [relu(x), relu(-x)], then for s = 1..nu the products
      r * (r rolled left by s), concatenated in order of s.
    * "poly2": the degree-2 polynomial map of "Transformers are RNNs"
      sec. 3.2.1, the outer product x x^T flattened row by row.
    sumnorm divides each feature vector by the sum of its components.
    """
    x = _as64(x)
    if fm == "elu1":
        f = phi_np(x)
    elif fm == "dpfp":
        r = np.concatenate([np.maximum(x, 0.0), np.maximum(-x, 0.0)], axis=-1)
        f = np.concatenate([r * np.roll(r, -s, axis=-1) for s in range(1, nu + 1)], axis=-1)
    elif fm == "poly2":
        D = x.shape[-1]
        f = (x[..., :, None] * x[..., None, :]).reshape(x.shape[:-1] + (D * D,))
    else:
        raise ValueError(fm)
    if sumnorm:
        f = f / f.sum(axis=-1, keepdims=True)
    return f


def definition_variant(q, k, v, fm: str, nu: int = 1, norm: str = "den", causal: bool = True) -> np.ndarray:
    """Quadratic form of a sum-update variant: w_ij = phi(q_i)^T phi(k_j)
    (eq. (4) with the variant's phi), masked to j <= i when causal (eq. (8));
    "den" divides by sum_j w_ij (eq. (3)), "sum" uses sum-normalised features
    and no denominator, "none" no denominator."""
    v = _as64(v)
    sn = norm == "sum"
    w = features_np(q, fm, nu, sn) @ np.swapaxes(features_np(k, fm, nu, sn), -1, -2)
    if causal:
        N = w.shape[-1]
        w = w * np.tril(np.ones((N, N)))
    out = w @ v
    if norm == "den":
        out = out / w.sum(axis=-1, keepdims=True)
    return out
