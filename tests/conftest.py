import os
import sys

import pytest

# the fault-injection tests set the library's test options, which a process
# must opt in to
os.environ.setdefault("DSEQ_ENABLE_TEST_OPTIONS", "1")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size case, minutes of oracle time")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.load()
