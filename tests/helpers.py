"""Shared test helpers: the error measure and tolerances.

Error measure (the pages give none; this reading is stated in the design
notes): per output row, max_m |y - r| / max_m |r|, maximised over all rows.
An element-wise relative error is ill-posed because outputs are averages of
zero-mean values and pass near 0.  The same per-head measure is used for the
final state S (per head) and z.
"""
import numpy as np
import torch

TOL_F32 = 1e-4     # fp32 inputs, fp32 arithmetic
TOL_BF16 = 2e-2    # bf16 operands on tensor cores, fp32 accumulation and state


def to64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def row_rel_err(y, r):
    """max over rows of max|y - r| / max|r| along the last axis."""
    y, r = to64(y), to64(r)
    assert y.shape == r.shape, (y.shape, r.shape)
    if y.size == 0:
        return 0.0
    num = np.abs(y - r).max(axis=-1)
    den = np.abs(r).max(axis=-1)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max())


def head_rel_err(y, r, nlead=2):
    """Same measure with everything after the first `nlead` axes flattened (states)."""
    y, r = to64(y), to64(r)
    return row_rel_err(y.reshape(y.shape[:nlead] + (-1,)), r.reshape(r.shape[:nlead] + (-1,)))


def tol_for(dtype):
    return TOL_F32 if dtype == torch.float32 else TOL_BF16


def sample_rows(N, C, count, seed):
    """Rows to check on long sequences: first, chunk edges, last, plus seeded picks."""
    rng = np.random.default_rng(seed)
    fixed = [0, 1, C - 1, C, C + 1, N // 2, N - 2, N - 1]
    picks = rng.integers(0, N, size=max(0, count - len(fixed)))
    rows = np.unique(np.clip(np.array(fixed + list(picks)), 0, N - 1))
    return rows
