import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmie.so")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    # all host cores: rows and heads are independent and each keeps its serial sum, so
    # the oracle's results are the same bits as on one thread (pinned by a test)
    oracle.set_threads(oracle.max_threads())
    return oracle
