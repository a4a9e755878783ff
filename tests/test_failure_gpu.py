"""Failure detection on the GPU without faulting it.

Every wait inside the tensor-core kernels is bounded.  The library's test hook
makes the next causal launch wait on an mbarrier that nothing arrives on, with
a ~2 ms limit; the kernel must give up, record LA_ERR_TIMEOUT in the device
error word, free its TMEM and return, leaving the context usable.
"""
import pytest
import torch

import oracle
from tests.helpers import TOL_BF16, row_rel_err
from weight_recurrence_gb300 import inputs, la

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    la.lib()


def test_injected_wait_timeout_is_reported_and_recoverable():
    q, k, v = inputs.qkv(1, 2, 300, 64, 64, torch.bfloat16, 0.125, seed=11)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert la.la_get_last_error() == la.LA_OK
    la.la_debug_inject_timeout(True, 2000)
    try:
        la.la_forward_causal(qd, kd, vd)
        st = la.la_get_last_error()
    finally:
        la.la_debug_inject_timeout(False)
    assert st == la.LA_ERR_TIMEOUT
    # the word was cleared and the context still works
    assert la.la_get_last_error() == la.LA_OK
    out = la.la_forward_causal(qd, kd, vd)
    assert la.la_get_last_error() == la.LA_OK
    assert row_rel_err(out, oracle.causal(q, k, v)[0]) <= TOL_BF16
