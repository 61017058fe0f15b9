import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes of CPU oracle work)")


def golden_path(name):
    return os.path.join(ROOT, "tests", "golden", name)


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle
