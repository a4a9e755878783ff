"""Seeded random shapes through the forward and backward entry points, against the fp64 oracle.

The other GPU tests pick their shapes by hand (chunk edges, ragged tails,
segment splits, full-size workloads).  Here a fixed seed draws batch, heads,
sequence length (1 to 2500: one chunk or many, ragged), head sizes D, M from
{16, 32, 64, 128}, dtype, input scale and whether a state is carried in,
so that routes and tile counts are mixed in ways no hand-picked case covers:
the tensor-core kernels (bf16 with D, M in {64, 128}), the CUDA-core ones
(fp32, or the smaller sizes), segments, clusters and the decode step.  The
error measure and tolerances are those of every parity test (1e-4 fp32,
2e-2 bf16, per-row, tests/helpers.py).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import head_rel_err, row_rel_err, tol_for
from weight_recurrence_gb300 import inputs, la

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SIZES = (16, 32, 64, 128)


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.lib()
    oracle.build()


def _draw(i):
    """Case i of the sweep: (B, H, N, D, M, dtype, scale, carry)."""
    rng = np.random.default_rng(4242 + i)
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    N = int(rng.choice([1, int(rng.integers(2, 129)), int(rng.integers(129, 2501))]))
    D, M = int(rng.choice(SIZES)), int(rng.choice(SIZES))
    # bf16 twice as often, and then the tensor-core sizes half of the time
    dtype = torch.bfloat16 if rng.random() < 2 / 3 else torch.float32
    if dtype == torch.bfloat16 and rng.random() < 0.5:
        D, M = int(rng.choice((64, 128))), int(rng.choice((64, 128)))
    scale = float(rng.choice([0.125, 0.5, 1.0])) / (1.0 if D <= 64 else 2.0)
    carry = bool(rng.random() < 0.5)
    return B, H, N, D, M, dtype, scale, carry


CASES = list(range(40))


@pytest.mark.parametrize("i", CASES)
def test_causal_random_shapes(i):
    B, H, N, D, M, dtype, scale, carry = _draw(i)
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=7000 + i)
    S0, z0 = inputs.state(B, H, D, M, seed=7100 + i, scale=0.05) if carry else (None, None)
    S = S0.clone().to(DEV) if carry else torch.zeros(B, H, D, M, device=DEV)
    z = z0.clone().to(DEV) if carry else torch.zeros(B, H, D, device=DEV)
    out = la.la_forward_causal(q.to(DEV), k.to(DEV), v.to(DEV), S=S, z=z)
    assert la.la_get_last_error() == la.LA_OK
    ref, Sr, zr = oracle.causal(q, k, v, S0, z0)
    tol = tol_for(dtype)
    assert row_rel_err(out, ref) <= tol, (B, H, N, D, M, dtype, carry)
    assert head_rel_err(S, Sr) <= tol and head_rel_err(z, zr) <= tol, (B, H, N, D, M, dtype, carry)


@pytest.mark.parametrize("i", CASES)
def test_noncausal_random_shapes(i):
    B, H, N, D, M, dtype, scale, _ = _draw(i)
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=7200 + i)
    out = la.la_forward_noncausal(q.to(DEV), k.to(DEV), v.to(DEV))
    assert la.la_get_last_error() == la.LA_OK
    assert row_rel_err(out, oracle.noncausal(q, k, v)[0]) <= tol_for(dtype), (B, H, N, D, M, dtype)


@pytest.mark.parametrize("i", CASES[:20])
def test_decode_random_shapes(i):
    B, H, _, D, M, dtype, scale, _ = _draw(i)
    steps = 1 + i % 5
    S0, z0 = inputs.state(B, H, D, M, seed=7300 + i, scale=0.05)
    qs, ks, vs = inputs.decode_tokens(steps, B, H, D, M, dtype, seed=7400 + i, scale=scale)
    S, z = S0.clone().to(DEV), z0.clone().to(DEV)
    Sr, zr = S0.double().numpy().copy(), z0.double().numpy().copy()
    for t in range(steps):
        y = la.la_decode_step(qs[t].to(DEV), ks[t].to(DEV), vs[t].to(DEV), S, z)
        yr = oracle.decode_step(qs[t], ks[t], vs[t], Sr, zr)
        assert row_rel_err(y, yr) <= tol_for(dtype), (B, H, D, M, dtype, t)
    assert la.la_get_last_error() == la.LA_OK
    assert head_rel_err(S, Sr) <= tol_for(dtype) and head_rel_err(z, zr) <= tol_for(dtype)


def _draw_bwd(i):
    """Backward case i: as _draw, with the tensor-core sizes (bf16, D, M in
    {64, 128}) half of the time and long sequences (up to 1500 rows, several
    chunks) more often."""
    rng = np.random.default_rng(9100 + i)
    B, H = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    N = int(rng.choice([1, int(rng.integers(2, 129)), int(rng.integers(129, 1501)), int(rng.integers(129, 1501))]))
    if rng.random() < 0.5:
        dtype, D, M = torch.bfloat16, int(rng.choice((64, 128))), int(rng.choice((64, 128)))
    else:
        dtype = torch.bfloat16 if rng.random() < 0.5 else torch.float32
        D, M = int(rng.choice(SIZES)), int(rng.choice(SIZES))
    scale = float(rng.choice([0.125, 0.5, 1.0])) / (1.0 if D <= 64 else 2.0)
    carry = bool(rng.random() < 0.5)
    return B, H, N, D, M, dtype, scale, carry


def _grad_err(y, r, G):
    """Per head: max |y - r| / max(max |r|, 1e-3 max |dout|) (the backward tests' measure)."""
    y = y.detach().float().cpu().numpy().astype(np.float64)
    r = np.asarray(r, np.float64)
    lead = y.shape[:2]
    y, r = y.reshape(lead + (-1,)), r.reshape(lead + (-1,))
    g = np.abs(G.float().numpy().astype(np.float64)).reshape(lead + (-1,)).max(axis=-1)
    den = np.maximum(np.abs(r).max(axis=-1), 1e-3 * g)
    den = np.where(den == 0, 1.0, den)
    return float((np.abs(y - r).max(axis=-1) / den).max())


@pytest.mark.parametrize("i", CASES[:24])
def test_causal_backward_random_shapes(i):
    """Random shapes through la_backward_causal (the two-sweep, segmented and CUDA-core routes), with a
    carried-in state and a final-state gradient half of the time."""
    B, H, N, D, M, dtype, scale, carry = _draw_bwd(i)
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=7500 + i)
    G = torch.randn((B, H, N, M), generator=torch.Generator().manual_seed(7600 + i)).to(dtype)
    if carry:
        S0, z0 = inputs.state(B, H, D, M, seed=7700 + i, scale=0.05)
        dSN, dzN = inputs.state(B, H, D, M, seed=7800 + i, scale=0.001)
        dS0 = torch.empty(B, H, D, M, device=DEV)
        dz0 = torch.empty(B, H, D, device=DEV)
        got = la.la_backward_causal(q.to(DEV), k.to(DEV), v.to(DEV), G.to(DEV), S0=S0.to(DEV), z0=z0.to(DEV),
                                    dSN=dSN.to(DEV), dzN=dzN.to(DEV), dS0=dS0, dz0=dz0)
        ref = oracle.causal_backward(q, k, v, G, S0=S0, z0=z0, dSN=dSN, dzN=dzN)
    else:
        got = la.la_backward_causal(q.to(DEV), k.to(DEV), v.to(DEV), G.to(DEV))
        ref = oracle.causal_backward(q, k, v, G)
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    tol = tol_for(dtype)
    for name, g, r in zip(("dq", "dk", "dv"), got, ref[:3]):
        assert _grad_err(g, r, G) <= tol, (name, B, H, N, D, M, dtype, carry)
    if carry:
        assert head_rel_err(dS0.cpu(), ref[3]) <= 2e-2 and head_rel_err(dz0.cpu(), ref[4]) <= 2e-2


@pytest.mark.parametrize("i", CASES[:16])
def test_noncausal_backward_random_shapes(i):
    B, H, N, D, M, dtype, scale, _ = _draw_bwd(100 + i)
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=7900 + i)
    G = torch.randn((B, H, N, M), generator=torch.Generator().manual_seed(8000 + i)).to(dtype)
    got = la.la_backward_noncausal(q.to(DEV), k.to(DEV), v.to(DEV), G.to(DEV))
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    for name, g, r in zip(("dq", "dk", "dv"), got, oracle.noncausal_backward(q, k, v, G)):
        assert _grad_err(g, r, G) <= tol_for(dtype), (name, B, H, N, D, M, dtype)
