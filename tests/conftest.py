import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _device_error_word_clear(request):
    """After every GPU test, the library's device error word must be clear: a
    bounded wait that gave up (LA_ERR_TIMEOUT) or, in the checked build, an
    access caught outside a buffer (LA_ERR_BOUNDS) that the test did not
    itself expect and read fails the test, whatever its results."""
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    from weight_recurrence_gb300 import la
    if la._lib is None:
        return
    st = la.la_get_last_error()
    assert st == la.LA_OK, "device error word after the test: %s" % la.status_string(st)
