"""The allocation-free non-causal entry point (collected last on purpose).

la_forward_noncausal_noalloc serves callers that cannot allocate device
memory (they get pointers from a framework that owns the memory pool, or run
a loop that must not call the allocator).  Its partial sums live in a fixed
8 MiB array inside the library.  This test calls it twice in a row through
the C ABI and checks each result against la_forward_noncausal (which uses a
caller workspace) and against the fp64 oracle, within the bf16 / fp32
tolerances of the other tests.  One case is large enough that the array
holds fewer key splits than the workspace entry point would use, so the
capped split count is exercised too.
"""
import ctypes

import pytest
import torch

import oracle
from tests.helpers import row_rel_err, tol_for
from weight_recurrence_gb300 import inputs, la

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.lib()
    oracle.build()


def _call_noalloc(q, k, v, out):
    s = la.shape_of(q, v)
    st = la.lib().la_forward_noncausal_noalloc(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                               ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()), s,
                                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st


@pytest.mark.parametrize("B,H,N,D,M,dtype", [(2, 4, 1000, 64, 64, torch.bfloat16),
                                             (1, 3, 777, 128, 128, torch.bfloat16),
                                             (2, 2, 300, 32, 64, torch.float32),
                                             # 16 heads x (128*128 + 128) floats = 1.06 MB per key
                                             # split: the array holds 7 splits, fewer than the 16
                                             # the workspace entry point picks for N = 4096
                                             (4, 4, 4096, 128, 128, torch.bfloat16)])
def test_noalloc_matches_workspace_entry_point_twice(B, H, N, D, M, dtype):
    outs = []
    for seed in (123, 124):   # two calls in a row, different data
        qh, kh, vh = inputs.qkv(B, H, N, D, M, dtype, 0.25, seed=seed)
        q, k, v = qh.cuda(), kh.cuda(), vh.cuda()
        ref = la.la_forward_noncausal(q, k, v)
        out = torch.full_like(ref, float("nan"))
        assert _call_noalloc(q, k, v, out) == la.LA_OK
        torch.cuda.synchronize()
        assert la.la_get_last_error() == la.LA_OK
        assert row_rel_err(out, ref) <= tol_for(dtype)
        exact, _, _ = oracle.noncausal(qh, kh, vh)
        assert row_rel_err(out, exact) <= tol_for(dtype)
        outs.append(out)
    assert not torch.equal(outs[0], outs[1])


def test_noalloc_rejects_problems_beyond_the_scratch():
    # B*H*(D*M + D)*4 bytes > 8 MiB: rejected on the host before any launch
    B, H, N, D, M = 1, 200, 16, 128, 128
    q = torch.zeros(B, H, N, D, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(B, H, N, M, dtype=torch.bfloat16, device="cuda")
    assert _call_noalloc(q, q.clone(), q.clone(), out) == la.LA_ERR_UNSUPPORTED
