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
