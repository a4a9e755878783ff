"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Every case draws seeded inputs from weight_recurrence_gb300.inputs, runs the
library on cuda:0, and compares with the oracle on the same values:
fp32 inputs within 1e-4, bf16 inputs within 2e-2 (per-row relative measure,
tests/helpers.py).  Every case compares every output element with the
recurrence oracle (the full decode workload: six replayed heads); small
cases and sampled rows of the full-size workloads are also compared with the
definition form.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import definition_causal, definition_rows
from tests.helpers import TOL_BF16, TOL_F32, head_rel_err, row_rel_err, sample_rows, to64, tol_for
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


# ------------------------------------------------------------------ causal

CAUSAL_CASES = [
    # (B, H, N, D, M, dtype, scale, chunk)
    (1, 1, 64, 16, 16, torch.float32, 1.0, 0),       # the tiny fp32 workload
    (2, 3, 1, 16, 32, torch.float32, 1.0, 0),
    (1, 2, 37, 32, 16, torch.float32, 1.0, 0),
    (2, 1, 300, 64, 64, torch.float32, 0.5, 0),
    (1, 1, 257, 128, 128, torch.float32, 1.0 / math.sqrt(128), 0),
    (1, 2, 129, 128, 16, torch.float32, 1.0, 0),
    (2, 3, 1000, 64, 64, torch.bfloat16, 0.125, 0),
    (2, 2, 1000, 64, 64, torch.bfloat16, 0.125, 64),
    (2, 2, 1000, 64, 64, torch.bfloat16, 0.125, 128),
    (1, 2, 515, 128, 128, torch.bfloat16, 1.0 / math.sqrt(128), 0),
    (1, 2, 300, 64, 128, torch.bfloat16, 0.125, 0),
    (1, 2, 300, 128, 64, torch.bfloat16, 0.125, 0),
    (2, 2, 127, 64, 64, torch.bfloat16, 1.0, 0),
    (1, 3, 200, 16, 32, torch.bfloat16, 1.0, 0),
    (1, 1, 1, 64, 64, torch.bfloat16, 1.0, 0),
    # large inputs (|x| up to ~20): phi's exponential far from 0 on the tensor path
    (2, 2, 700, 64, 64, torch.bfloat16, 4.0, 0),
    (1, 2, 400, 128, 128, torch.bfloat16, 3.0, 0),
    (1, 2, 300, 64, 128, torch.bfloat16, 5.0, 0),
    # long sequences with few heads: split into segments (two-pass state carry)
    (1, 2, 5000, 64, 64, torch.bfloat16, 0.125, 0),
    (1, 1, 9000, 128, 128, torch.bfloat16, 1.0 / math.sqrt(128), 0),
    (1, 1, 4100, 64, 128, torch.bfloat16, 0.125, 0),
]


@pytest.mark.parametrize("B,H,N,D,M,dtype,scale,chunk", CAUSAL_CASES)
def test_causal_vs_oracle(B, H, N, D, M, dtype, scale, chunk):
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=B * 1000 + N + D + M)
    ref, Sref, zref = oracle.causal(q, k, v)
    qd, kd, vd = _dev(q, k, v)
    S = torch.zeros(B, H, D, M, device=DEV)
    z = torch.zeros(B, H, D, device=DEV)
    out = la.la_forward_causal(qd, kd, vd, chunk=chunk, S=S, z=z)
    torch.cuda.synchronize()
    tol = tol_for(dtype)
    assert row_rel_err(out, ref) <= tol
    assert head_rel_err(S, Sref) <= tol
    assert head_rel_err(z, zref) <= tol
    if N <= 300:
        assert row_rel_err(out, definition_causal(q, k, v)) <= tol


@pytest.mark.parametrize("dtype,D,M,N", [(torch.float32, 32, 64, 333), (torch.bfloat16, 64, 64, 333),
                                         (torch.bfloat16, 128, 128, 333), (torch.bfloat16, 64, 64, 6000),
                                         (torch.bfloat16, 128, 64, 3500)])
def test_causal_state_carry_in_and_out(dtype, D, M, N):
    B, H = 1, 2
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, 1.0 / math.sqrt(D), seed=77)
    S0, z0 = inputs.state(B, H, D, M, seed=78)
    ref, Sref, zref = oracle.causal(q, k, v, S0=S0.double().numpy(), z0=z0.double().numpy())
    qd, kd, vd = _dev(q, k, v)
    S, z = _dev(S0.clone(), z0.clone())
    out = la.la_forward_causal(qd, kd, vd, S=S, z=z)
    torch.cuda.synchronize()
    tol = tol_for(dtype)
    assert row_rel_err(out, ref) <= tol
    assert head_rel_err(S, Sref) <= tol
    assert head_rel_err(z, zref) <= tol


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_causal_state_only(dtype):
    B, H, N, D, M = 1, 4, 700, 64, 64
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, 0.125, seed=79)
    _, Sref, zref = oracle.causal(q, k, v, want_out=False)
    qd, kd, vd = _dev(q, k, v)
    S = torch.zeros(B, H, D, M, device=DEV)
    z = torch.zeros(B, H, D, device=DEV)
    la.la_forward_causal(qd, kd, vd, S=S, z=z, want_out=False)
    torch.cuda.synchronize()
    assert head_rel_err(S, Sref) <= tol_for(dtype)
    assert head_rel_err(z, zref) <= tol_for(dtype)


@pytest.mark.parametrize("split", [1, 63, 64, 200])
def test_causal_split_equals_whole(split):
    """causal(X) = causal(X[:n]) then causal(X[n:], carried state) (sec. 3.3.2)."""
    B, H, N, D, M = 1, 2, 400, 64, 64
    q, k, v = _dev(*inputs.qkv(B, H, N, D, M, torch.bfloat16, 0.125, seed=80))
    whole = la.la_forward_causal(q, k, v)
    S = torch.zeros(B, H, D, M, device=DEV)
    z = torch.zeros(B, H, D, device=DEV)
    a = la.la_forward_causal(q[:, :, :split].contiguous(), k[:, :, :split].contiguous(),
                             v[:, :, :split].contiguous(), S=S, z=z)
    b = la.la_forward_causal(q[:, :, split:].contiguous(), k[:, :, split:].contiguous(),
                             v[:, :, split:].contiguous(), S=S, z=z)
    torch.cuda.synchronize()
    assert row_rel_err(torch.cat([a, b], dim=2), whole) <= TOL_BF16


def test_causal_empty_sequence_keeps_state():
    D = M = 64
    q = torch.empty(1, 2, 0, D, dtype=torch.bfloat16, device=DEV)
    S0, z0 = _dev(*inputs.state(1, 2, D, M, seed=5))
    S, z = S0.clone(), z0.clone()
    out = la.la_forward_causal(q, q, q, S=S, z=z)
    torch.cuda.synchronize()
    assert out.shape == (1, 2, 0, M)
    assert torch.equal(S, S0) and torch.equal(z, z0)


def test_chunk_length_invariance():
    B, H, N, D, M = 2, 2, 777, 64, 64
    q, k, v = _dev(*inputs.qkv(B, H, N, D, M, torch.bfloat16, 0.125, seed=81))
    outs = [la.la_forward_causal(q, k, v, chunk=c) for c in (0, 64, 128)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert row_rel_err(o, outs[0]) <= TOL_BF16


def test_constant_v_reproduces_itself():
    B, H, N, D, M = 1, 2, 500, 64, 64
    q, k, _ = inputs.qkv(B, H, N, D, M, torch.bfloat16, 1.0, seed=82)
    v = torch.full((B, H, N, M), 1.5, dtype=torch.bfloat16)
    v[..., 1::2] = -0.75
    qd, kd, vd = _dev(q, k, v)
    out = la.la_forward_causal(qd, kd, vd)
    nc = la.la_forward_noncausal(qd, kd, vd)
    torch.cuda.synchronize()
    assert row_rel_err(out, v) <= 4e-3
    assert row_rel_err(nc, v) <= 4e-3


def test_last_causal_row_equals_noncausal():
    B, H, N, D, M = 2, 2, 600, 64, 64
    q, k, v = _dev(*inputs.qkv(B, H, N, D, M, torch.bfloat16, 0.125, seed=83))
    c = la.la_forward_causal(q, k, v)
    n = la.la_forward_noncausal(q, k, v)
    torch.cuda.synchronize()
    assert row_rel_err(c[:, :, -1], n[:, :, -1]) <= TOL_BF16


def test_prefix_independence():
    B, H, N, D, M = 1, 2, 500, 64, 64
    q, k, v = inputs.qkv(B, H, N, D, M, torch.bfloat16, 0.125, seed=84)
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[:, :, 300:] += 1
    k2[:, :, 300:] -= 1
    v2[:, :, 300:] *= 2
    o1 = la.la_forward_causal(*_dev(q, k, v))
    o2 = la.la_forward_causal(*_dev(q2, k2, v2))
    torch.cuda.synchronize()
    # rows before the change see exactly the same data; chunking may differ only
    # beyond the first changed chunk, so compare the rows of whole unchanged chunks
    assert torch.equal(o1[:, :, :256], o2[:, :, :256])


# --------------------------------------------------------------- non-causal

NC_CASES = [
    (1, 1, 64, 16, 16, torch.float32, 1.0),
    (2, 3, 1, 32, 16, torch.float32, 1.0),
    (2, 2, 1000, 64, 64, torch.float32, 0.5),
    (1, 2, 300, 128, 128, torch.float32, 1.0 / math.sqrt(128)),
    (2, 3, 1000, 64, 64, torch.bfloat16, 1.0),
    (1, 2, 4099, 128, 128, torch.bfloat16, 1.0 / math.sqrt(128)),
    (2, 2, 333, 64, 128, torch.bfloat16, 1.0),
    (1, 2, 200, 128, 64, torch.bfloat16, 1.0),
    (2, 2, 100, 16, 64, torch.bfloat16, 1.0),
    # large inputs on the tensor path
    (2, 2, 700, 64, 64, torch.bfloat16, 4.0),
    (1, 2, 500, 128, 128, torch.bfloat16, 5.0),
    (1, 2, 333, 128, 64, torch.bfloat16, 3.0),
]


@pytest.mark.parametrize("B,H,N,D,M,dtype,scale", NC_CASES)
def test_noncausal_vs_oracle(B, H, N, D, M, dtype, scale):
    q, k, v = inputs.qkv(B, H, N, D, M, dtype, scale, seed=2000 + N + D)
    ref, _, _ = oracle.noncausal(q, k, v)
    out = la.la_forward_noncausal(*_dev(q, k, v))
    torch.cuda.synchronize()
    assert row_rel_err(out, ref) <= tol_for(dtype)


# ------------------------------------------- back-to-back dependent launches

def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


def test_back_to_back_calls_read_the_previous_output():
    """Each call reads the output of the call just before it, with no host
    synchronisation in between: the launches overlap their set-up with the
    previous launch's tail, and their first global reads must still see that
    launch's writes.  The oracle runs the same chain on its own outputs
    (rounded to bf16 as the library's are)."""
    B, H, N, D = 2, 4, 700, 64
    q, k, v = inputs.qkv(B, H, N, D, D, torch.bfloat16, 1.0, seed=95)
    qd, kd, vd = _dev(q, k, v)
    o1 = la.la_forward_causal(qd, kd, vd)
    o2 = la.la_forward_noncausal(o1, kd, vd)
    o3 = la.la_forward_causal(qd, o2, vd)
    o4 = la.la_forward_noncausal(o3, o3, o1)
    torch.cuda.synchronize()
    r1 = _bf16(oracle.causal(q, k, v)[0])
    r2 = _bf16(oracle.noncausal(r1, k, v)[0])
    r3 = _bf16(oracle.causal(q, r2, v)[0])
    r4 = oracle.noncausal(r3, r3, r1)[0]
    assert row_rel_err(o3, r3) <= TOL_BF16
    assert row_rel_err(o4, r4) <= TOL_BF16


def test_back_to_back_decode_steps_feed_their_outputs_forward():
    """Decode steps whose query is the previous step's output, issued back to
    back (the state is read and rewritten in place by every step)."""
    B, H, D, steps = 3, 4, 64, 6
    S0, z0 = inputs.state(B, H, D, D, seed=96)
    _, ks, vs = inputs.decode_tokens(steps, B, H, D, D, torch.bfloat16, seed=97)
    q0 = inputs.decode_tokens(1, B, H, D, D, torch.bfloat16, seed=98)[0][0]
    S, z = _dev(S0.clone(), z0.clone())
    ys, y = [], q0.to(DEV)
    for t in range(steps):
        y = la.la_decode_step(y, *_dev(ks[t], vs[t]), S, z)
        ys.append(y)
    torch.cuda.synchronize()
    Sr, zr = S0.double().numpy().copy(), z0.double().numpy().copy()
    yr = q0
    for t in range(steps):
        yr = _bf16(oracle.decode_step(yr, ks[t], vs[t], Sr, zr))
        assert row_rel_err(ys[t], yr) <= TOL_BF16
    assert head_rel_err(S, Sr) <= 1e-5


# ------------------------------------------------------------------- decode

@pytest.mark.parametrize("dtype,D,M", [(torch.float32, 16, 16), (torch.float32, 64, 64),
                                       (torch.bfloat16, 64, 64), (torch.bfloat16, 128, 128),
                                       (torch.bfloat16, 32, 128), (torch.bfloat16, 128, 16)])
def test_decode_vs_oracle(dtype, D, M):
    B, H, steps = 3, 5, 12
    S0, z0 = inputs.state(B, H, D, M, seed=90)
    qs, ks, vs = inputs.decode_tokens(steps, B, H, D, M, dtype, seed=91)
    Sr, zr = S0.double().numpy().copy(), z0.double().numpy().copy()
    S, z = _dev(S0.clone(), z0.clone())
    tol = tol_for(dtype)
    for t in range(steps):
        yr = oracle.decode_step(qs[t], ks[t], vs[t], Sr, zr)
        y = la.la_decode_step(*_dev(qs[t], ks[t], vs[t]), S, z)
        torch.cuda.synchronize()
        assert row_rel_err(y, yr) <= tol
    assert head_rel_err(S, Sr) <= (1e-5 if dtype == torch.float32 else 1e-5)
    assert head_rel_err(z, zr) <= 1e-5


def test_prefill_then_decode_equals_causal():
    """The decoder continues exactly where the causal forward leaves its state."""
    B, H, N, D, M, T = 2, 3, 200, 64, 64, 8
    q, k, v = inputs.qkv(B, H, N + T, D, M, torch.bfloat16, 1.0, seed=92)
    ref, _, _ = oracle.causal(q, k, v)
    qd, kd, vd = _dev(q, k, v)
    S = torch.zeros(B, H, D, M, device=DEV)
    z = torch.zeros(B, H, D, device=DEV)
    la.la_forward_causal(qd[:, :, :N].contiguous(), kd[:, :, :N].contiguous(), vd[:, :, :N].contiguous(),
                         S=S, z=z, want_out=False)
    for t in range(T):
        y = la.la_decode_step(qd[:, :, N + t].contiguous(), kd[:, :, N + t].contiguous(),
                              vd[:, :, N + t].contiguous(), S, z)
        torch.cuda.synchronize()
        assert row_rel_err(y, ref[:, :, N + t]) <= TOL_BF16


def test_decode_from_zero_state_returns_v():
    B, H, D, M = 4, 4, 64, 64
    qs, ks, vs = inputs.decode_tokens(1, B, H, D, M, torch.bfloat16, seed=93)
    S = torch.zeros(B, H, D, M, device=DEV)
    z = torch.zeros(B, H, D, device=DEV)
    y = la.la_decode_step(*_dev(qs[0], ks[0], vs[0]), S, z)
    torch.cuda.synchronize()
    assert row_rel_err(y, vs[0]) <= 4e-3


# ------------------------------------------------------ full-size workloads

def _row_err_by_head(out, ref):
    """row_rel_err over [BH, N, M] arrays, one head at a time (bounded host memory)."""
    worst = 0.0
    for i in range(out.shape[0]):
        worst = max(worst, row_rel_err(out[i], ref[i]))
    return worst


def _full_causal(w, chunk=None, spot_heads=3, spot_rows=24):
    """The full workload in the bench's launch configuration, every element:
    all rows of all heads against the fp64 recurrence (eqs. (10)-(12)), every
    head's final S and z, and a few sampled rows against the independent
    definition form (eq. (9))."""
    q, k, v = inputs.workload_inputs(w)
    qd, kd, vd = _dev(q, k, v)
    S = torch.zeros(w.B, w.H, w.D, w.M, device=DEV)
    z = torch.zeros(w.B, w.H, w.D, device=DEV)
    out = la.la_forward_causal(qd, kd, vd, chunk=w.chunk if chunk is None else chunk, S=S, z=z)
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    del qd, kd, vd
    out = out.cpu().reshape(w.B * w.H, w.N, w.M)
    ref, Sref, zref = oracle.causal(q, k, v)
    err = _row_err_by_head(out, ref.reshape(w.B * w.H, w.N, w.M))
    assert err <= TOL_BF16, err
    assert head_rel_err(S.cpu(), Sref) <= TOL_BF16
    assert head_rel_err(z.cpu(), zref) <= TOL_BF16
    del ref
    rng = np.random.default_rng(w.seed)
    flat = [(b, h) for b in range(w.B) for h in range(w.H)]
    worst = 0.0
    for idx in rng.choice(len(flat), size=min(spot_heads, len(flat)), replace=False):
        b, h = flat[idx]
        rows = sample_rows(w.N, 128, spot_rows, seed=int(idx))
        d = definition_rows(q[b, h], k[b, h], v[b, h], rows, True)
        worst = max(worst, row_rel_err(out[b * w.H + h][rows], d))
    assert worst <= TOL_BF16, worst


def test_full_causal_b16h8n3072d64():
    """Every output element of B16 H8 N3072 D64 at the configured chunk hint (64)."""
    _full_causal(inputs.WORKLOADS["causal_b16h8n3072d64"])


def test_full_causal_b16h8n3072d64_default_chunk():
    _full_causal(inputs.WORKLOADS["causal_b16h8n3072d64"], chunk=0, spot_heads=1)


def test_full_causal_b1h16n65536d128():
    """Every output element of the long workload (segments carried through the
    segment-sum pre-pass)."""
    _full_causal(inputs.WORKLOADS["causal_b1h16n65536d128"], spot_heads=2, spot_rows=16)


def test_full_causal_b16h8n3072d64_three_calls_back_to_back():
    """Three full-size calls issued back to back with no host synchronisation,
    each continuing from the state the previous one left (consecutive
    segments of one 9216-token sequence).  Each launch overlaps its set-up
    (and its L2 prefetch of its first tiles) with the previous launch's tail;
    every element of all three outputs and the final state are compared with
    the recurrence over the whole sequence."""
    w = inputs.WORKLOADS["causal_b16h8n3072d64"]
    parts = [inputs.qkv(w.B, w.H, w.N, w.D, w.M, w.dtype, w.scale, seed=w.seed + 100 * (i + 1))
             for i in range(3)]
    S = torch.zeros(w.B, w.H, w.D, w.M, device=DEV)
    z = torch.zeros(w.B, w.H, w.D, device=DEV)
    devs = [_dev(*p) for p in parts]
    outs = [torch.empty(w.B, w.H, w.N, w.M, dtype=w.dtype, device=DEV) for _ in range(3)]
    torch.cuda.synchronize()
    for (qd, kd, vd), o in zip(devs, outs):
        la.la_forward_causal(qd, kd, vd, out=o, chunk=w.chunk, S=S, z=z)
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    del devs
    q, k, v = (torch.cat([p[j] for p in parts], dim=2) for j in range(3))
    ref, Sref, zref = oracle.causal(q, k, v)
    out = torch.cat([o.cpu() for o in outs], dim=2).reshape(w.B * w.H, 3 * w.N, w.M)
    err = _row_err_by_head(out, ref.reshape(w.B * w.H, 3 * w.N, w.M))
    assert err <= TOL_BF16, err
    assert head_rel_err(S.cpu(), Sref) <= TOL_BF16
    assert head_rel_err(z.cpu(), zref) <= TOL_BF16


def test_full_noncausal_b8h8n4096d64():
    w = inputs.WORKLOADS["noncausal_b8h8n4096d64"]
    q, k, v = inputs.workload_inputs(w)
    out = la.la_forward_noncausal(*_dev(q, k, v))
    torch.cuda.synchronize()
    ref, _, _ = oracle.noncausal(q, k, v)
    assert row_rel_err(out, ref) <= TOL_BF16


def test_full_tiny_f32_vs_definition():
    w = inputs.WORKLOADS["causal_tiny_f32"]
    q, k, v = inputs.workload_inputs(w)
    out = la.la_forward_causal(*_dev(q, k, v))
    torch.cuda.synchronize()
    assert row_rel_err(out, definition_causal(q, k, v)) <= TOL_F32


def test_full_decode_b256h16d64():
    """The full decode workload in the bench's launch configuration: a 1024-token
    prefill through the causal forward, then 4096 sequential steps over the whole
    [256, 16] batch.  Sampled heads are replayed by the recurrence oracle; their
    outputs are compared at steps 0, 1, 2, 1023, every 512th and 4095, and their
    final state after the last step."""
    w = inputs.WORKLOADS["decode_b256h16d64"]
    B, H, D, M, T = w.B, w.H, w.D, w.M, w.steps
    q, k, v = inputs.workload_inputs(w)
    rng = np.random.default_rng(w.seed)
    flat = rng.choice(B * H, size=6, replace=False)
    bsel, hsel = torch.as_tensor(flat // H), torch.as_tensor(flat % H)
    S = torch.zeros(B, H, D, M, device=DEV)
    z = torch.zeros(B, H, D, device=DEV)
    la.la_forward_causal(*_dev(q, k, v), S=S, z=z, want_out=False)
    _, Sr, zr = oracle.causal(q[bsel, hsel], k[bsel, hsel], v[bsel, hsel], want_out=False)
    del q, k, v
    qs, ks, vs = inputs.decode_tokens(T, B, H, D, M, w.dtype, seed=inputs.rank_seed(w.seed + 1000, 0), device=DEV)
    check = sorted({0, 1, 2, 1023, T - 1} | set(range(0, T, 512)))
    y = torch.empty(B, H, M, dtype=w.dtype, device=DEV)
    seen = {}
    bd, hd = bsel.to(DEV), hsel.to(DEV)
    for t in range(T):
        la.la_decode_step(qs[t], ks[t], vs[t], S, z, y=y)
        if t in check:
            seen[t] = y[bd, hd].clone()
    torch.cuda.synchronize()
    assert la.la_get_last_error() == la.LA_OK
    qh, kh, vh = (x[:, bd, hd].cpu() for x in (qs, ks, vs))
    del qs, ks, vs
    worst = 0.0
    for t in range(T):
        yr = oracle.decode_step(qh[t], kh[t], vh[t], Sr, zr, nthreads=1)
        if t in seen:
            worst = max(worst, row_rel_err(seen[t].cpu(), yr))
    assert worst <= TOL_BF16, worst
    assert head_rel_err(S[bd, hd].cpu(), Sr, nlead=1) <= TOL_BF16
    assert head_rel_err(z[bd, hd].cpu(), zr, nlead=1) <= TOL_BF16
