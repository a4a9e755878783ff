"""The bounds-checked build (liblinattn_checked.so) on the GPU.

The checked build compiles the release kernels with a check in front of each
global access whose index comes from run-time values (workspace slots,
carried-in state rows, per-sequence lengths, direct output rows); a failed
check skips the access and records LA_ERR_BOUNDS.  These tests

* run the paths that carry checks -- the causal tensor-core kernel with and
  without the segment-sum pre-pass and with a carried-in state, the
  non-causal tensor-core kernel with both exchanges (cluster shared memory at
  D = M = 64, the workspace at D = M = 128), the CUDA-core fp32 paths and the
  allocation-free entry point -- through the checked library, and require
  LA_OK and the oracle's result: no check fires on a correct call;
* turn on the library's own injection hook, which offsets a state row or a
  workspace slot past its buffer inside the kernel, and require
  LA_ERR_BOUNDS; the check caught the index before the access, so the next
  call on the same context is LA_OK and correct again.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import head_rel_err, row_rel_err, tol_for
from weight_recurrence_gb300 import inputs, la

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def checked_lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    oracle.build()
    prev = la.lib()
    L = la.select_library(True)
    assert la.la_checked_build()
    yield L
    la.la_debug_inject_bounds(False)
    la._lib = prev


def _err():
    torch.cuda.synchronize()
    return la.la_get_last_error()


# (B, H, N, D, M, dtype): a ragged tail in every case; B*H = 2 at N = 8192
# splits each head into segments (pre-pass + workspace loads)
CAUSAL = [(2, 2, 300, 64, 64, torch.bfloat16),
          (1, 2, 8192, 64, 64, torch.bfloat16),
          (1, 2, 4100, 128, 128, torch.bfloat16),
          (2, 2, 200, 32, 64, torch.float32)]


@pytest.mark.parametrize("B,H,N,D,M,dtype", CAUSAL)
def test_causal_with_state_is_clean_and_exact(B, H, N, D, M, dtype):
    qh, kh, vh = inputs.qkv(B, H, N, D, M, dtype, 0.25, seed=31)
    S0, z0 = inputs.state(B, H, D, M, seed=32)
    S, z = S0.to(DEV), z0.to(DEV)
    out = la.la_forward_causal(qh.to(DEV), kh.to(DEV), vh.to(DEV), S=S, z=z)
    assert _err() == la.LA_OK
    ref, Sr, zr = oracle.causal(qh, kh, vh, S0, z0)
    tol = tol_for(dtype)
    assert row_rel_err(out, ref) <= tol
    assert head_rel_err(S, Sr) <= tol and head_rel_err(z, zr) <= tol


def test_causal_varlen_is_clean():
    B, H, N, D, M = 3, 2, 520, 64, 64
    qh, kh, vh = inputs.qkv(B, H, N, D, M, torch.bfloat16, 0.25, seed=33)
    lens = torch.tensor([520, 129, 1], dtype=torch.int32)
    out = la.la_forward_causal_varlen(qh.to(DEV), kh.to(DEV), vh.to(DEV), lens.to(DEV))
    assert _err() == la.LA_OK
    for b, n in enumerate(lens.tolist()):
        ref, _, _ = oracle.causal(qh[b:b + 1, :, :n], kh[b:b + 1, :, :n], vh[b:b + 1, :, :n])
        assert row_rel_err(out[b:b + 1, :, :n], ref) <= tol_for(torch.bfloat16)


@pytest.mark.parametrize("B,H,N,D,M,dtype", [(2, 4, 1000, 64, 64, torch.bfloat16),
                                             (1, 3, 777, 128, 128, torch.bfloat16),
                                             (2, 2, 300, 32, 64, torch.float32)])
@pytest.mark.parametrize("noalloc", [False, True])
def test_noncausal_is_clean_and_exact(B, H, N, D, M, dtype, noalloc):
    qh, kh, vh = inputs.qkv(B, H, N, D, M, dtype, 0.25, seed=34)
    fn = la.la_forward_noncausal_noalloc if noalloc else la.la_forward_noncausal
    out = fn(qh.to(DEV), kh.to(DEV), vh.to(DEV))
    assert _err() == la.LA_OK
    ref, _, _ = oracle.noncausal(qh, kh, vh)
    assert row_rel_err(out, ref) <= tol_for(dtype)


def _injected(call):
    la.la_debug_inject_bounds(True)
    try:
        call()
        return _err()
    finally:
        la.la_debug_inject_bounds(False)


@pytest.mark.parametrize("N", [300, 8192])   # one segment; segments and the pre-pass
def test_injected_state_index_is_caught(N):
    B, H, D, M = 1, 2, 64, 64
    qh, kh, vh = inputs.qkv(B, H, N, D, M, torch.bfloat16, 0.25, seed=35)
    S0, z0 = inputs.state(B, H, D, M, seed=36)
    q, k, v = qh.to(DEV), kh.to(DEV), vh.to(DEV)
    assert _injected(lambda: la.la_forward_causal(q, k, v, S=S0.to(DEV), z=z0.to(DEV))) == la.LA_ERR_BOUNDS
    # the context is intact: the same call without the hook is clean and exact
    S, z = S0.to(DEV), z0.to(DEV)
    out = la.la_forward_causal(q, k, v, S=S, z=z)
    assert _err() == la.LA_OK
    ref, Sr, _ = oracle.causal(qh, kh, vh, S0, z0)
    assert row_rel_err(out, ref) <= tol_for(torch.bfloat16)
    assert head_rel_err(S, Sr) <= tol_for(torch.bfloat16)


def test_injected_workspace_slot_is_caught_in_noalloc():
    B, H, N, D, M = 2, 2, 300, 32, 64
    qh, kh, vh = inputs.qkv(B, H, N, D, M, torch.float32, 0.25, seed=37)
    q, k, v = qh.to(DEV), kh.to(DEV), vh.to(DEV)
    assert _injected(lambda: la.la_forward_noncausal_noalloc(q, k, v)) == la.LA_ERR_BOUNDS
    out = la.la_forward_noncausal_noalloc(q, k, v)
    assert _err() == la.LA_OK
    assert row_rel_err(out, oracle.noncausal(qh, kh, vh)[0]) <= tol_for(torch.float32)


def test_release_build_ignores_the_hook():
    release = la.select_library(False)
    try:
        assert not la.la_checked_build()
        qh, kh, vh = inputs.qkv(1, 2, 300, 64, 64, torch.bfloat16, 0.25, seed=38)
        S = torch.zeros(1, 2, 64, 64, device=DEV)
        z = torch.zeros(1, 2, 64, device=DEV)
        la.la_debug_inject_bounds(True)
        out = la.la_forward_causal(qh.to(DEV), kh.to(DEV), vh.to(DEV), S=S, z=z)
        la.la_debug_inject_bounds(False)
        assert _err() == la.LA_OK
        assert row_rel_err(out, oracle.causal(qh, kh, vh)[0]) <= tol_for(torch.bfloat16)
    finally:
        assert la.select_library(True) is not release
    assert np.isfinite(out.float().cpu().numpy()).all()


@pytest.mark.parametrize("D,M", [(64, 128), (128, 128)])
def test_segmented_causal_backward_is_clean_and_exact(D, M):
    """The segmented tensor-core causal backward (segment key sums, scans, query
    and key passes) through the checked build, with a carried-in state and a
    final-state gradient: no check fires and the results are the oracle's."""
    B, H, N = 1, 2, 1500   # one head cut into several segments
    qh, kh, vh = inputs.qkv(B, H, N, D, M, torch.bfloat16, 0.125, seed=41)
    G = torch.randn((B, H, N, M), generator=torch.Generator().manual_seed(42)).to(torch.bfloat16)
    S0, z0 = inputs.state(B, H, D, M, seed=43, scale=0.05)
    dSN, dzN = inputs.state(B, H, D, M, seed=44, scale=0.001)
    dS0 = torch.empty(B, H, D, M, device=DEV)
    dz0 = torch.empty(B, H, D, device=DEV)
    got = la.la_backward_causal(qh.to(DEV), kh.to(DEV), vh.to(DEV), G.to(DEV), S0=S0.to(DEV), z0=z0.to(DEV),
                                dSN=dSN.to(DEV), dzN=dzN.to(DEV), dS0=dS0, dz0=dz0)
    assert _err() == la.LA_OK
    ref = oracle.causal_backward(qh, kh, vh, G, S0=S0, z0=z0, dSN=dSN, dzN=dzN)
    for g, r in zip(got, ref[:3]):
        y = g.float().cpu().numpy().astype(np.float64).reshape(B * H, -1)
        rr = np.asarray(r, np.float64).reshape(B * H, -1)
        den = np.maximum(np.abs(rr).max(axis=-1), 1e-3 * float(G.float().abs().max()))
        assert float((np.abs(y - rr).max(axis=-1) / den).max()) <= 2e-2
    assert head_rel_err(dS0.cpu(), ref[3]) <= 2e-2 and head_rel_err(dz0.cpu(), ref[4]) <= 2e-2


@pytest.mark.parametrize("D,M", [(64, 64), (128, 128)])
def test_noncausal_backward_is_clean_and_exact(D, M):
    """The tensor-core non-causal backward (key sums, query and key passes) through the checked build."""
    B, H, N = 1, 2, 700
    qh, kh, vh = inputs.qkv(B, H, N, D, M, torch.bfloat16, 0.25, seed=39)
    G = torch.randn((B, H, N, M), generator=torch.Generator().manual_seed(40)).to(torch.bfloat16)
    got = la.la_backward_noncausal(qh.to(DEV), kh.to(DEV), vh.to(DEV), G.to(DEV))
    assert _err() == la.LA_OK
    ref = oracle.noncausal_backward(qh, kh, vh, G)
    for g, r in zip(got, ref):
        y = g.float().cpu().numpy().astype(np.float64).reshape(B * H, -1)
        rr = np.asarray(r, np.float64).reshape(B * H, -1)
        den = np.maximum(np.abs(rr).max(axis=-1), 1e-3 * float(G.float().abs().max()))
        assert float((np.abs(y - rr).max(axis=-1) / den).max()) <= 2e-2
    # the key-sum pass offsets its workspace slot past the workspace: caught
    qd, kd, vd, Gd = qh.to(DEV), kh.to(DEV), vh.to(DEV), G.to(DEV)
    assert _injected(lambda: la.la_backward_noncausal(qd, kd, vd, Gd)) == la.LA_ERR_BOUNDS
