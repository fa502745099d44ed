import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for _p in (ROOT, TESTS):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size parity case")


@pytest.fixture(scope="session")
def orc():
    from oracle import Oracle
    return Oracle()


@pytest.fixture(scope="session")
def orc_mt():
    """The same oracle source built with OpenMP: the full-size parity cases
    compare every output element, which the single-threaded build cannot
    finish in the test's time."""
    from oracle import Oracle
    return Oracle(threads=True)
