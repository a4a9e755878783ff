"""GPU parity of the backward pass (through the C ABI) against the fp64 oracle.

Error measure: per head, max |y - r| / max(max |r|, 1e-3 max |dout|) over the
head's gradient tensor.  A gradient row can be far smaller than the terms
that cancel in it (so the per-row measure of the forward is too strict), and
some gradients vanish exactly (one token: the output is V whatever Q and K
are), so the denominator has a floor tied to the size of the incoming
gradient.  Tolerances as the forward's: 1e-4 for fp32, 2e-2 for bf16 tensors.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import head_rel_err
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


def _tol(dtype):
    return 1e-4 if dtype == torch.float32 else 2e-2


def _dout(B, H, N, M, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn((B, H, N, M), generator=g).to(dtype).contiguous()


def _dev(*ts):
    return [None if t is None else t.to(DEV) for t in ts]


def grad_err(y, r, G, nlead=2):
    y = y.detach().float().cpu().numpy().astype(np.float64)
    r = np.asarray(r, np.float64)
    G = np.asarray(G.float().cpu().numpy() if hasattr(G, "cpu") else G, np.float64)
    lead = y.shape[:nlead]
    y, r, G = y.reshape(lead + (-1,)), r.reshape(lead + (-1,)), G.reshape(lead + (-1,))
    den = np.maximum(np.abs(r).max(axis=-1), 1e-3 * np.abs(G).max(axis=-1))
    den = np.where(den == 0, 1.0, den)
    return float((np.abs(y - r).max(axis=-1) / den).max())


def _check_grads(got, ref, dtype, G, what=""):
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        err = grad_err(g, r, G)
        assert err <= _tol(dtype), (what, name, err)


CASES = [
    # (B, H, N, D, M, dtype, scale)
    (1, 1, 64, 16, 16, torch.float32, 1.0),
    (2, 3, 1, 16, 32, torch.float32, 1.0),
    (1, 2, 37, 32, 16, torch.float32, 1.0),
    (2, 1, 300, 64, 64, torch.float32, 0.5),
    (1, 1, 129, 128, 128, torch.float32, 1.0 / math.sqrt(128)),
    (2, 2, 1000, 64, 64, torch.bfloat16, 0.125),
    (1, 2, 515, 128, 128, torch.bfloat16, 1.0 / math.sqrt(128)),
    (1, 2, 300, 64, 128, torch.bfloat16, 0.125),
    (1, 3, 200, 128, 16, torch.bfloat16, 1.0),
    # tensor-core path (bf16, D = M = 64): ragged, shorter than a chunk, one chunk
    (1, 2, 77, 64, 64, torch.bfloat16, 0.125),
    (2, 1, 128, 64, 64, torch.bfloat16, 1.0),
    (1, 3, 645, 64, 64, torch.bfloat16, 0.5),
    # two chunks exactly, and a last chunk of one row (the sweeps prepare the
    # next chunk's feature maps while the current one's products run)
    (1, 2, 256, 64, 64, torch.bfloat16, 0.25),
    (2, 1, 129, 64, 64, torch.bfloat16, 0.25),
]


@pytest.mark.parametrize("B,H,N,D,M,dtype,scale", CASES)
def test_causal_backward_vs_oracle(B, H, N, D, M, dtype, scale):
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=500 + N)
    G = _dout(B, H, N, M, dtype, 600 + N)
    ref = oracle.causal_backward(q, k, v, G)[:3]
    got = la.la_backward_causal(*_dev(q, k, v, G))
    torch.cuda.synchronize()
    _check_grads(got, ref, dtype, G, "causal")


@pytest.mark.parametrize("B,H,N,D,M,dtype,scale", CASES)
def test_noncausal_backward_vs_oracle(B, H, N, D, M, dtype, scale):
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=700 + N)
    G = _dout(B, H, N, M, dtype, 800 + N)
    ref = oracle.noncausal_backward(q, k, v, G)
    got = la.la_backward_noncausal(*_dev(q, k, v, G))
    torch.cuda.synchronize()
    _check_grads(got, ref, dtype, G, "noncausal")


@pytest.mark.parametrize("dtype,D,M", [(torch.float32, 32, 64), (torch.bfloat16, 32, 64), (torch.bfloat16, 64, 64),
                                       (torch.bfloat16, 128, 128), (torch.bfloat16, 64, 128),
                                       (torch.bfloat16, 128, 64)])
def test_causal_backward_with_state(dtype, D, M):
    """Carried-in state, gradient through the final state, and dS0/dz0 out
    (bf16 with D, M >= 64: the tensor-core paths, sequential and chunked)."""
    B, H, N = 2, 2, 150 if D == M == 64 else 400
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, 0.25, seed=901)
    G = _dout(B, H, N, M, dtype, 902)
    S0, z0 = inputs.state(B, H, D, M, seed=903, scale=0.05)
    dSN, dzN = inputs.state(B, H, D, M, seed=904, scale=0.001)
    dzN = dzN * 1e-3
    rq, rk, rv, rS, rz = oracle.causal_backward(q, k, v, G, S0=S0, z0=z0, dSN=dSN, dzN=dzN)
    dS0 = torch.empty(B, H, D, M, device=DEV)
    dz0 = torch.empty(B, H, D, device=DEV)
    qd, kd, vd, Gd, S0d, z0d, dSNd, dzNd = _dev(q, k, v, G, S0, z0, dSN, dzN)
    got = la.la_backward_causal(qd, kd, vd, Gd, S0=S0d, z0=z0d, dSN=dSNd, dzN=dzNd, dS0=dS0, dz0=dz0)
    torch.cuda.synchronize()
    _check_grads(got, (rq, rk, rv), dtype, G, "state")
    tc = dtype == torch.bfloat16 and D >= 64
    assert head_rel_err(dS0.cpu(), rS) <= (2e-2 if tc else 1e-4)
    assert head_rel_err(dz0.cpu(), rz) <= (2e-2 if tc else 1e-4)


@pytest.mark.parametrize("B,H,N,D,M", [(16, 4, 2000, 128, 128),    # two segments of eight chunks per head
                                       (16, 8, 1000, 64, 128)])    # one segment per head
def test_segmented_backward_with_state_many_heads(B, H, N, D, M):
    """Carried-in state and final-state gradient on the segmented route with
    several chunks per segment (the state carried along the segment in TMEM)
    and with one segment per head (no segment key sums: the scan only copies
    the carried-in state)."""
    dtype = torch.bfloat16
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, 0.125, seed=905)
    G = _dout(B, H, N, M, dtype, 906)
    S0, z0 = inputs.state(B, H, D, M, seed=907, scale=0.05)
    dSN, dzN = inputs.state(B, H, D, M, seed=908, scale=0.001)
    rq, rk, rv, rS, rz = oracle.causal_backward(q, k, v, G, S0=S0, z0=z0, dSN=dSN, dzN=dzN)
    dS0 = torch.empty(B, H, D, M, device=DEV)
    dz0 = torch.empty(B, H, D, device=DEV)
    qd, kd, vd, Gd, S0d, z0d, dSNd, dzNd = _dev(q, k, v, G, S0, z0, dSN, dzN)
    got = la.la_backward_causal(qd, kd, vd, Gd, S0=S0d, z0=z0d, dSN=dSNd, dzN=dzNd, dS0=dS0, dz0=dz0)
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    _check_grads(got, (rq, rk, rv), dtype, G, "segmented state")
    assert head_rel_err(dS0.cpu(), rS) <= 2e-2 and head_rel_err(dz0.cpu(), rz) <= 2e-2


@pytest.mark.parametrize("dtype,D,M", [(torch.float32, 64, 64), (torch.bfloat16, 64, 64),
                                       (torch.bfloat16, 128, 128)])
def test_causal_backward_split_chains(dtype, D, M):
    """Backward of two segments joined through dS0 -> dSN equals the whole backward."""
    B, H, N, split = 1, 2, 333, 130
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, 0.125, seed=910)
    G = _dout(B, H, N, M, dtype, 911)
    qd, kd, vd, Gd = _dev(q, k, v, G)
    whole = la.la_backward_causal(qd, kd, vd, Gd)
    S1 = torch.zeros(B, H, D, M, device=DEV)
    z1 = torch.zeros(B, H, D, device=DEV)
    la.la_forward_causal(qd[:, :, :split].contiguous(), kd[:, :, :split].contiguous(),
                         vd[:, :, :split].contiguous(), S=S1, z=z1, want_out=False)
    dS1 = torch.empty(B, H, D, M, device=DEV)
    dz1 = torch.empty(B, H, D, device=DEV)
    sl2 = [t[:, :, split:].contiguous() for t in (qd, kd, vd, Gd)]
    g2 = la.la_backward_causal(*sl2, S0=S1, z0=z1, dS0=dS1, dz0=dz1)
    sl1 = [t[:, :, :split].contiguous() for t in (qd, kd, vd, Gd)]
    g1 = la.la_backward_causal(*sl1, dSN=dS1, dzN=dz1)
    torch.cuda.synchronize()
    for a, b, w in zip(g1, g2, whole):
        assert grad_err(torch.cat([a, b], dim=2), w.float().cpu().numpy(), G) <= _tol(dtype)


def test_causal_backward_empty_passes_state_gradient_through():
    B, H, D, M = 2, 3, 16, 16
    q = torch.empty(B, H, 0, D, device=DEV)
    v = torch.empty(B, H, 0, M, device=DEV)
    dSN = torch.randn(B, H, D, M, device=DEV)
    dzN = torch.randn(B, H, D, device=DEV)
    dS0 = torch.full((B, H, D, M), 7.0, device=DEV)
    dz0 = torch.full((B, H, D), 7.0, device=DEV)
    la.la_backward_causal(q, q, v, v, dSN=dSN, dzN=dzN, dS0=dS0, dz0=dz0)
    torch.cuda.synchronize()
    assert torch.equal(dS0, dSN) and torch.equal(dz0, dzN)


def test_causal_backward_constant_v():
    """Constant V: every output is that constant, so dQ and dK vanish."""
    B, H, N, D, M = 1, 2, 200, 32, 32
    q, k, _ = inputs.qkv(B, H, N, D, M, torch.float32, 0.5, seed=920)
    v = torch.full((B, H, N, M), 0.75)
    G = _dout(B, H, N, M, torch.float32, 921)
    dq, dk, dv = la.la_backward_causal(*_dev(q, k, v, G))
    torch.cuda.synchronize()
    assert dq.abs().max().item() < 1e-5 * G.abs().max().item()
    assert dk.abs().max().item() < 1e-5 * G.abs().max().item()


def test_full_causal_backward_b16h8n3072d64():
    """The training-shaped workload at full size; sampled heads against the oracle."""
    w = inputs.WORKLOADS["causal_b16h8n3072d64"]
    q, k, v = inputs.workload_inputs(w)
    G = _dout(w.B, w.H, w.N, w.M, w.dtype, 930)
    dq, dk, dv = la.la_backward_causal(*_dev(q, k, v, G))
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    rng = np.random.default_rng(931)
    for idx in rng.choice(w.B * w.H, size=4, replace=False):
        b, h = divmod(int(idx), w.H)
        ref = oracle.causal_backward(q[b, h][None], k[b, h][None], v[b, h][None], G[b, h][None])[:3]
        for got, r in zip((dq, dk, dv), ref):
            assert grad_err(got[b, h][None], r, G[b, h][None], nlead=1) <= 2e-2


# Segmented causal backward on tensor cores (bf16, D, M in {64, 128} other
# than D = M = 64): one row, shorter than a chunk, one chunk exactly, a last
# chunk of one row, many chunks with a ragged tail, all three (D, M); heads
# cut into one-chunk segments (few heads) and into several chunks each.
CHUNK_TC_CASES = [
    (1, 1, 1, 128, 128, 1.0 / math.sqrt(128)),
    (1, 2, 77, 128, 128, 1.0 / math.sqrt(128)),
    (2, 1, 128, 64, 128, 0.25),
    (1, 2, 129, 128, 64, 1.0 / math.sqrt(128)),
    (1, 2, 1000, 128, 128, 1.0 / math.sqrt(128)),
    (2, 2, 3000, 64, 128, 0.125),
    (1, 1, 4097, 128, 64, 1.0),
    (16, 4, 2000, 128, 128, 1.0 / math.sqrt(128)),
    (64, 4, 700, 64, 128, 0.25),
]


@pytest.mark.parametrize("B,H,N,D,M,scale", CHUNK_TC_CASES)
def test_causal_backward_chunked_tensor_cores(B, H, N, D, M, scale):
    dtype = torch.bfloat16
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=1300 + N)
    G = _dout(B, H, N, M, dtype, 1400 + N)
    ref = oracle.causal_backward(q, k, v, G)[:3]
    n0 = la.la_launch_count()
    got = la.la_backward_causal(*_dev(q, k, v, G))
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    # [segment key sums,] forward scan, query pass, reverse scan, key pass; the
    # key sums run only when a head is cut into several segments (about one
    # CTA per SM)
    nch = (N + 127) // 128
    nseg = max(1, min(nch, torch.cuda.get_device_properties(0).multi_processor_count // (B * H)))
    assert la.la_launch_count() - n0 == (5 if nseg > 1 else 4)
    _check_grads(got, ref, dtype, G, "causal chunked tc")


def test_full_causal_backward_b1h16n65536d128():
    """The long-context shape (D = M = 128) at full size; sampled heads against the oracle."""
    w = inputs.WORKLOADS["causal_b1h16n65536d128"]
    q, k, v = inputs.workload_inputs(w)
    G = _dout(w.B, w.H, w.N, w.M, w.dtype, 950)
    dq, dk, dv = la.la_backward_causal(*_dev(q, k, v, G))
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    rng = np.random.default_rng(951)
    for h in rng.choice(w.H, size=2, replace=False):
        h = int(h)
        ref = oracle.causal_backward(q[0, h][None], k[0, h][None], v[0, h][None], G[0, h][None])[:3]
        for got, r in zip((dq, dk, dv), ref):
            assert grad_err(got[0, h][None], r, G[0, h][None], nlead=1) <= 2e-2


# Non-causal backward on tensor cores (bf16, D, M in {64, 128}): key ranges
# split across CTAs (several ranges per head, ragged last chunk, a range
# shorter than a chunk), all four (D, M) pairs.
NC_TC_CASES = [
    (1, 1, 1, 64, 64, 1.0),
    (1, 2, 100, 64, 64, 0.5),
    (2, 3, 1300, 64, 64, 0.125),
    (1, 2, 4000, 64, 64, 1.0),
    (1, 1, 777, 64, 128, 0.25),
    (1, 2, 640, 128, 64, 1.0 / math.sqrt(128)),
    (2, 1, 1025, 128, 128, 1.0 / math.sqrt(128)),
]


@pytest.mark.parametrize("B,H,N,D,M,scale", NC_TC_CASES)
def test_noncausal_backward_tensor_cores(B, H, N, D, M, scale):
    dtype = torch.bfloat16
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=1100 + N)
    G = _dout(B, H, N, M, dtype, 1200 + N)
    ref = oracle.noncausal_backward(q, k, v, G)
    n0 = la.la_launch_count()
    got = la.la_backward_noncausal(*_dev(q, k, v, G))
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    assert la.la_launch_count() - n0 == 3      # key sums, query kernel, key kernel
    _check_grads(got, ref, dtype, G, "noncausal tc")


def test_full_noncausal_backward_b16h8n3072d64():
    """The training-shaped shape at full size, every element against the oracle."""
    w = inputs.WORKLOADS["causal_b16h8n3072d64"]
    q, k, v = inputs.workload_inputs(w)
    G = _dout(w.B, w.H, w.N, w.M, w.dtype, 940)
    got = la.la_backward_noncausal(*_dev(q, k, v, G))
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    ref = oracle.noncausal_backward(q, k, v, G)
    _check_grads(got, ref, w.dtype, G, "noncausal full")
