"""GPU parity of batched stateful generation (through the C ABI) against the oracle:
a prefill of sequences of different lengths (la_forward_causal_varlen) and
several recurrent steps in one launch (la_decode_steps), "Transformers are
RNNs" sec. 3.3-3.4 (eqs. (10)-(12), (18)-(20)) applied per sequence."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import TOL_BF16, head_rel_err, row_rel_err, tol_for
from weight_recurrence_gb300 import inputs
from weight_recurrence_gb300 import la

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.lib()
    oracle.build()


def _dev(*ts):
    return [t.to(DEV) for t in ts]


@pytest.mark.parametrize("dtype,D,M", [(torch.float32, 32, 16), (torch.bfloat16, 64, 64),
                                       (torch.bfloat16, 128, 128), (torch.bfloat16, 64, 128)])
def test_varlen_prefill_vs_oracle(dtype, D, M):
    B, H, N = 4, 2, 700
    lens = [700, 1, 0, 333]
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, 0.25, seed=1100 + D)
    S0, z0 = inputs.state(B, H, D, M, seed=1101, scale=0.01)
    S, z = _dev(S0.clone(), z0.clone())
    out = la.la_forward_causal_varlen(*_dev(q, k, v), torch.tensor(lens, dtype=torch.int32, device=DEV),
                                      S=S, z=z)
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    tol = tol_for(dtype)
    for b, n in enumerate(lens):
        if n > 0:
            ref, Sr, zr = oracle.causal(q[b, :, :n], k[b, :, :n], v[b, :, :n], S0=S0[b], z0=z0[b])
            assert row_rel_err(out[b, :, :n], ref) <= tol
        else:
            Sr, zr = S0[b].double().numpy(), z0[b].double().numpy()
        assert head_rel_err(S[b].cpu(), Sr, nlead=1) <= tol
        assert head_rel_err(z[b].cpu(), zr, nlead=1) <= tol


def test_varlen_full_lengths_equal_uniform_call():
    B, H, N, D, M = 2, 3, 400, 64, 64
    q, k, v = _dev(*inputs.qkv(B, H, N, D, M, torch.bfloat16, 0.125, seed=1110))
    a = la.la_forward_causal(q, k, v)
    b = la.la_forward_causal_varlen(q, k, v, torch.full((B,), N, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("dtype,D,M", [(torch.float32, 32, 16), (torch.bfloat16, 64, 64),
                                       (torch.bfloat16, 128, 128), (torch.bfloat16, 128, 32)])
def test_decode_steps_vs_oracle(dtype, D, M):
    T, B, H = 37, 3, 4
    steps = [37, 5, 0]
    S0, z0 = inputs.state(B, H, D, M, seed=1120, scale=0.02)
    qs, ks, vs = inputs.decode_tokens(T, B, H, D, M, dtype, seed=1121)
    S, z = _dev(S0.clone(), z0.clone())
    y = torch.full((T, B, H, M), 9.0, dtype=dtype, device=DEV)
    la.la_decode_steps(*_dev(qs, ks, vs), S, z, y=y, steps=torch.tensor(steps, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    tol = tol_for(dtype)
    y = y.cpu()
    for b, n in enumerate(steps):
        Sr, zr = S0[b].double().numpy().copy(), z0[b].double().numpy().copy()
        for t in range(n):
            yr = oracle.decode_step(qs[t, b], ks[t, b], vs[t, b], Sr, zr)
            assert row_rel_err(y[t, b], yr) <= tol
        # the tensor-core path (bf16, D, M in {64, 128}) accumulates bf16 phi(K)
        stol = 1e-5 if dtype == torch.float32 or M == 32 else TOL_BF16
        assert head_rel_err(S[b].cpu(), Sr, nlead=1) <= stol
        assert head_rel_err(z[b].cpu(), zr, nlead=1) <= stol


def test_full_decode_steps_b256h16d64():
    """All 4096 steps of the decode workload in one launch; sampled heads against the oracle."""
    w = inputs.WORKLOADS["decode_b256h16d64"]
    B, H, D, M, T = w.B, w.H, w.D, w.M, w.steps
    rng = np.random.default_rng(w.seed + 7)
    flat = rng.choice(B * H, size=4, replace=False)
    bsel, hsel = torch.as_tensor(flat // H), torch.as_tensor(flat % H)
    S0, z0 = inputs.state(B, H, D, M, seed=1130, scale=0.01)
    qs, ks, vs = inputs.decode_tokens(T, B, H, D, M, w.dtype, seed=inputs.rank_seed(w.seed + 1000, 0), device=DEV)
    S, z = _dev(S0.clone(), z0.clone())
    y = la.la_decode_steps(qs, ks, vs, S, z)
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    bd, hd = bsel.to(DEV), hsel.to(DEV)
    qh, kh, vh, yh = (x[:, bd, hd].cpu() for x in (qs, ks, vs, y))
    Sr = S0[bsel, hsel].double().numpy().copy()
    zr = z0[bsel, hsel].double().numpy().copy()
    worst = 0.0
    for t in range(T):
        yr = oracle.decode_step(qh[t], kh[t], vh[t], Sr, zr, nthreads=1)
        if t % 64 == 0 or t == T - 1:
            worst = max(worst, row_rel_err(yh[t], yr))
    assert worst <= TOL_BF16
    assert head_rel_err(S[bd, hd].cpu(), Sr, nlead=1) <= TOL_BF16
