"""GPU parity of the variants (la_forward_causal_variant, la_forward_noncausal_variant,
la_decode_step_variant) through the C ABI against the fp64 variant oracle.

Feature maps DPFP-nu and degree-2 polynomial, sum-normalised features, the raw
read-out, and the delta update rule ("Linear Transformers Are Secretly Fast
Weight Programmers"; "Transformers are RNNs" sec. 3.2.1), on fp32 and bf16
inputs, ragged lengths, every instantiated feature width (F = 16 .. 512),
carried-in state, state-only calls, split-and-carry, decode steps, and the two
full-size variant workloads the bench times.  Tolerances as everywhere: 1e-4
for fp32 inputs, 2e-2 for bf16 (per-row relative measure, tests/helpers.py).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import head_rel_err, row_rel_err, to64, tol_for
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


def _start_state(B, H, F, M, norm, seed):
    """A random starting state: S ~ N(0, 1) / F, z > 0 (denominator only)."""
    g = torch.Generator().manual_seed(seed)
    S = torch.randn((B, H, F, M), generator=g) / F
    z = torch.rand((B, H, F), generator=g) + 0.5 if norm == "den" else None
    return S.contiguous(), (z.contiguous() if z is not None else None)


CASES = [
    # (fm, nu, norm, update, B, H, N, D, M, dtype, scale)
    ("elu1", 1, "den", "sum", 1, 2, 100, 16, 32, torch.float32, 1.0),
    ("elu1", 1, "den", "sum", 2, 2, 300, 64, 64, torch.bfloat16, 0.125),
    ("elu1", 1, "sum", "sum", 1, 2, 77, 32, 16, torch.float32, 1.0),
    ("elu1", 1, "none", "sum", 1, 1, 50, 16, 16, torch.float32, 1.0),
    ("dpfp", 1, "sum", "sum", 2, 2, 300, 64, 64, torch.bfloat16, 0.125),
    ("dpfp", 2, "none", "sum", 1, 2, 65, 16, 32, torch.float32, 1.0),
    ("dpfp", 3, "sum", "sum", 1, 2, 200, 64, 64, torch.bfloat16, 0.125),
    ("dpfp", 4, "sum", "sum", 1, 1, 40, 64, 16, torch.float32, 1.0),
    ("dpfp", 1, "sum", "sum", 1, 1, 33, 128, 128, torch.bfloat16, 1.0 / math.sqrt(128)),
    ("poly2", 1, "den", "sum", 1, 2, 100, 16, 16, torch.float32, 1.0),
    ("poly2", 1, "none", "sum", 1, 1, 70, 16, 64, torch.bfloat16, 0.5),
    ("elu1", 1, "sum", "delta", 1, 2, 100, 16, 16, torch.float32, 1.0),
    ("elu1", 1, "sum", "delta", 2, 2, 300, 64, 64, torch.bfloat16, 0.125),
    ("elu1", 1, "sum", "delta", 1, 1, 1, 128, 128, torch.bfloat16, 1.0),
    ("dpfp", 1, "sum", "delta", 1, 2, 129, 32, 32, torch.float32, 1.0),
    ("dpfp", 2, "sum", "delta", 1, 1, 257, 64, 128, torch.bfloat16, 0.125),
]


def _ids(c):
    return "%s%d-%s-%s-B%dH%dN%dD%dM%d-%s" % (c[0], c[1], c[2], c[3], c[4], c[5], c[6], c[7], c[8],
                                               "f32" if c[9] == torch.float32 else "bf16")


# bf16, sum update, F in {64, 128}: these run on the chunked tensor-core
# kernel, the feature map applied row by row on chip (elu + 1 also with the
# denominator, long enough that the plain form would split it into segments)
TC_CASES = [
    ("elu1", 1, "den", "sum", 1, 2, 9000, 64, 64, torch.bfloat16, 0.125),
    ("elu1", 1, "den", "sum", 2, 2, 1000, 64, 64, torch.bfloat16, 0.125),
    ("elu1", 1, "den", "sum", 1, 2, 300, 128, 128, torch.bfloat16, 1.0 / math.sqrt(128)),
    ("dpfp", 1, "sum", "sum", 2, 2, 1000, 64, 64, torch.bfloat16, 0.125),
    ("dpfp", 1, "none", "sum", 1, 2, 300, 64, 128, torch.bfloat16, 0.125),
    ("dpfp", 1, "sum", "sum", 1, 3, 257, 32, 64, torch.bfloat16, 0.25),
    ("dpfp", 2, "sum", "sum", 1, 2, 129, 16, 128, torch.bfloat16, 0.5),
    ("dpfp", 2, "none", "sum", 2, 1, 400, 32, 64, torch.bfloat16, 0.25),
    ("dpfp", 4, "sum", "sum", 1, 2, 200, 16, 128, torch.bfloat16, 0.5),
    ("elu1", 1, "sum", "sum", 2, 2, 777, 64, 64, torch.bfloat16, 0.125),
    ("elu1", 1, "sum", "sum", 1, 2, 300, 128, 128, torch.bfloat16, 1.0 / math.sqrt(128)),
    ("elu1", 1, "none", "sum", 1, 2, 300, 64, 128, torch.bfloat16, 0.125),
    ("elu1", 1, "none", "sum", 1, 1, 1, 128, 64, torch.bfloat16, 1.0),
    ("dpfp", 1, "sum", "sum", 1, 1, 1, 64, 64, torch.bfloat16, 0.125),
    # bf16 delta rule, F = M = 64: chunks of 128 tokens on tensor cores
    ("elu1", 1, "sum", "delta", 2, 2, 1000, 64, 64, torch.bfloat16, 0.125),
    ("elu1", 1, "sum", "delta", 1, 3, 3000, 64, 64, torch.bfloat16, 0.125),
    ("elu1", 1, "sum", "delta", 1, 2, 128, 64, 64, torch.bfloat16, 1.0),
    ("elu1", 1, "sum", "delta", 1, 1, 1, 64, 64, torch.bfloat16, 1.0),
    ("dpfp", 1, "sum", "delta", 2, 1, 777, 32, 64, torch.bfloat16, 0.25),
    ("dpfp", 2, "sum", "delta", 1, 2, 129, 16, 64, torch.bfloat16, 0.5),
    ("elu1", 1, "sum", "delta", 2, 1, 256, 64, 64, torch.bfloat16, 0.25),   # two chunks exactly
]


@pytest.mark.parametrize("case", CASES + TC_CASES, ids=_ids)
@pytest.mark.parametrize("with_state", [False, True])
def test_causal_variant_vs_oracle(case, with_state):
    fm, nu, norm, update, B, H, N, D, M, dtype, scale = case
    var = la.variant(fm, nu, norm, update)
    F = la.la_feature_dim(var, D)
    assert F == oracle.feature_dim(fm, D, nu)
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=N + D + M + nu)
    beta = inputs.betas(B, H, N, dtype, seed=N + 7) if update == "delta" else None
    S0, z0 = _start_state(B, H, F, M, norm, seed=N) if with_state else (None, None)
    ref, Sref, zref = oracle.variant_causal(q, k, v, fm, nu, norm, update, beta=beta, S0=S0, z0=z0)
    S = S0.clone().to(DEV) if with_state else torch.zeros(B, H, F, M, device=DEV)
    z = None
    if norm == "den":
        z = z0.clone().to(DEV) if with_state else torch.zeros(B, H, F, device=DEV)
    out = la.la_forward_causal_variant(q.to(DEV), k.to(DEV), v.to(DEV), var,
                                       beta=None if beta is None else beta.to(DEV), S=S, z=z)
    torch.cuda.synchronize()
    tol = tol_for(dtype)
    assert row_rel_err(out, ref) <= tol
    assert head_rel_err(S, Sref) <= tol
    if z is not None:
        assert head_rel_err(z, zref) <= tol


def test_variant_without_state_matches_zero_state():
    var = la.variant("dpfp", 1, "sum", "delta")
    q, k, v = inputs.qkv(2, 2, 90, 32, 32, torch.float32, 1.0, seed=31)
    beta = inputs.betas(2, 2, 90, torch.float32, seed=32)
    args = [t.to(DEV) for t in (q, k, v)]
    a = la.la_forward_causal_variant(*args, var, beta=beta.to(DEV))
    S = torch.zeros(2, 2, 128, 32, device=DEV)
    b = la.la_forward_causal_variant(*args, var, beta=beta.to(DEV), S=S)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("fm,nu,norm,update,D,M,dtype", [("elu1", 1, "den", "sum", 16, 32, torch.float32),
                                                         ("dpfp", 2, "sum", "delta", 16, 32, torch.float32),
                                                         ("poly2", 1, "none", "sum", 16, 32, torch.float32),
                                                         ("dpfp", 1, "sum", "sum", 64, 64, torch.bfloat16),
                                                         ("elu1", 1, "none", "sum", 64, 128, torch.bfloat16),
                                                         ("elu1", 1, "sum", "delta", 64, 64, torch.bfloat16)])
def test_state_only_and_split_carry(fm, nu, norm, update, D, M, dtype):
    """A state-only call (out = NULL) leaves the same state as a full call, and two
    calls chained through the state equal one call over the whole sequence (the
    bf16 cases run on the tensor-core kernel; their split is not chunk-aligned)."""
    B, H, N = 2, 2, 450
    var = la.variant(fm, nu, norm, update)
    F = la.la_feature_dim(var, D)
    q, k, v = [t.to(DEV) for t in inputs.qkv(B, H, N, D, M, dtype, 0.25, seed=41)]
    beta = inputs.betas(B, H, N, dtype, seed=42).to(DEV) if update == "delta" else None

    def state():
        return torch.zeros(B, H, F, M, device=DEV), (torch.zeros(B, H, F, device=DEV) if norm == "den" else None)

    Sw, zw = state()
    whole = la.la_forward_causal_variant(q, k, v, var, beta=beta, S=Sw, z=zw)
    So, zo = state()
    la.la_forward_causal_variant(q, k, v, var, beta=beta, S=So, z=zo, want_out=False)
    cut = 197
    Ss, zs = state()
    sl = lambda t, a, b: None if t is None else t[:, :, a:b].contiguous()
    first = la.la_forward_causal_variant(sl(q, 0, cut), sl(k, 0, cut), sl(v, 0, cut), var,
                                         beta=sl(beta, 0, cut), S=Ss, z=zs)
    second = la.la_forward_causal_variant(sl(q, cut, N), sl(k, cut, N), sl(v, cut, N), var,
                                          beta=sl(beta, cut, N), S=Ss, z=zs)
    torch.cuda.synchronize()
    tol = 1e-4 if dtype == torch.float32 else 2e-2
    assert head_rel_err(So, Sw) <= 1e-6
    assert row_rel_err(torch.cat([first, second], 2), whole) <= tol
    assert head_rel_err(Ss, Sw) <= tol


NC_CASES = [
    ("elu1", 1, "den", 2, 2, 500, 64, 64, torch.bfloat16, 1.0),
    ("elu1", 1, "sum", 1, 2, 130, 16, 32, torch.float32, 1.0),
    ("dpfp", 1, "sum", 2, 2, 700, 64, 64, torch.bfloat16, 0.125),
    ("dpfp", 3, "none", 1, 1, 90, 32, 16, torch.float32, 1.0),
    ("poly2", 1, "den", 1, 2, 333, 16, 128, torch.float32, 1.0),
    # bf16, F in {64, 128}: the one-launch tensor-core kernel
    ("elu1", 1, "den", 1, 2, 777, 128, 64, torch.bfloat16, 1.0 / math.sqrt(128)),
    ("dpfp", 1, "sum", 2, 3, 1000, 32, 128, torch.bfloat16, 0.25),
    ("dpfp", 4, "none", 1, 2, 257, 16, 64, torch.bfloat16, 0.5),
    ("elu1", 1, "sum", 2, 2, 3000, 64, 64, torch.bfloat16, 0.125),
    ("elu1", 1, "none", 1, 2, 129, 128, 128, torch.bfloat16, 1.0 / math.sqrt(128)),
    ("dpfp", 2, "sum", 1, 1, 1, 32, 64, torch.bfloat16, 0.25),
]


@pytest.mark.parametrize("fm,nu,norm,B,H,N,D,M,dtype,scale", NC_CASES)
def test_noncausal_variant_vs_oracle(fm, nu, norm, B, H, N, D, M, dtype, scale):
    var = la.variant(fm, nu, norm, "sum")
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=N + nu)
    ref = oracle.variant_noncausal(q, k, v, fm, nu, norm)
    out = la.la_forward_noncausal_variant(q.to(DEV), k.to(DEV), v.to(DEV), var)
    torch.cuda.synchronize()
    assert row_rel_err(out, ref) <= tol_for(dtype)


@pytest.mark.parametrize("fm,nu,norm,update,dtype", [("elu1", 1, "den", "sum", torch.float32),
                                                     ("dpfp", 1, "sum", "delta", torch.bfloat16),
                                                     ("poly2", 1, "none", "sum", torch.float32),
                                                     ("elu1", 1, "sum", "delta", torch.float32)])
def test_decode_variant_steps(fm, nu, norm, update, dtype):
    """Decode steps from a random state equal the oracle's causal rows over the
    same tokens started from that state (update, then read out)."""
    B, H, D, M, T = 3, 2, 16, 32, 5
    var = la.variant(fm, nu, norm, update)
    F = la.la_feature_dim(var, D)
    q, k, v = inputs.decode_tokens(T, B, H, D, M, dtype, seed=51)
    beta = inputs.betas(T, B, H, dtype, seed=52)
    S0, z0 = _start_state(B, H, F, M, norm, seed=53)
    # oracle: the T tokens as a sequence [B, H, T, .]
    seq = lambda x: x.permute(1, 2, 0, 3).contiguous()
    ref, Sref, zref = oracle.variant_causal(seq(q), seq(k), seq(v), fm, nu, norm, update,
                                            beta=beta.permute(1, 2, 0).contiguous() if update == "delta" else None,
                                            S0=S0, z0=z0)
    S = S0.clone().to(DEV)
    z = z0.clone().to(DEV) if z0 is not None else None
    ys = []
    for t in range(T):
        ys.append(la.la_decode_step_variant(q[t].to(DEV), k[t].to(DEV), v[t].to(DEV), S, var, z=z,
                                            beta=beta[t].to(DEV) if update == "delta" else None))
    torch.cuda.synchronize()
    y = torch.stack(ys, 2)
    tol = tol_for(dtype)
    assert row_rel_err(y, ref) <= tol
    assert head_rel_err(S, Sref) <= tol


@pytest.mark.parametrize("name", ["delta_b16h8n3072d64", "dpfp_b16h8n3072d64"])
def test_full_variant_workload(name):
    """The bench's variant workloads at full size, in its launch configuration;
    8 of the 128 heads replayed by the oracle (every row and the final state)."""
    w = inputs.WORKLOADS[name]
    fm, nu, norm, update = w.variant
    var = la.variant(fm, nu, norm, update)
    F = la.la_feature_dim(var, w.D)
    q, k, v = inputs.workload_inputs(w)
    beta = inputs.workload_betas(w) if update == "delta" else None
    S = torch.zeros(w.B, w.H, F, w.M, device=DEV)
    out = la.la_forward_causal_variant(q.to(DEV), k.to(DEV), v.to(DEV), var,
                                       beta=None if beta is None else beta.to(DEV), S=S)
    torch.cuda.synchronize()
    heads = [(0, 0), (3, 5), (7, 7), (8, 1), (11, 2), (13, 6), (15, 0), (15, 7)]
    for b, h in heads:
        sl = lambda t: t[b:b + 1, h:h + 1]
        ref, Sref, _ = oracle.variant_causal(sl(q), sl(k), sl(v), fm, nu, norm, update,
                                             beta=None if beta is None else sl(beta))
        assert row_rel_err(out[b:b + 1, h:h + 1], ref) <= tol_for(w.dtype), (b, h)
        assert head_rel_err(S[b:b + 1, h:h + 1], Sref) <= tol_for(w.dtype), (b, h)
