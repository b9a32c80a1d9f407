import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libfa.so")


@pytest.fixture(autouse=True)
def _parity_report_context():
    """Each test starts without the previous test's workload description in parity reports."""
    from tests import parity

    parity._context.clear()
    yield


@pytest.fixture(scope="session", autouse=True)
def _checked_build_records_no_violation():
    """With FA_CHECKED_BUILD=1 every test runs on libfa_debug.so, whose kernels check each global
    store against its tensor's extent; at the end of the session no violation may be recorded
    (the planted one of the bounds self-test is read and cleared by its own test)."""
    yield
    if os.environ.get("FA_CHECKED_BUILD") != "1":
        return
    import torch

    from tiled_online_softmax_gb300 import fa

    if not torch.cuda.is_available():
        return
    torch.cuda.synchronize()
    assert fa.bounds_report(fa.lib()) == (0, 0), "a kernel recorded an out-of-bounds store"
