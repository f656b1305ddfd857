import os
import sys

import pytest

TESTS = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(TESTS)
for _p in (ROOT, TESTS):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


@pytest.fixture(autouse=True)
def _parity_test_id(request):
    """Tag the parity records (tests/parity.py) with the running test."""
    import parity

    parity.CURRENT_TEST["id"] = request.node.nodeid
    yield


def pytest_sessionfinish(session, exitstatus):
    import parity

    parity.write_report()


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle
