import gc
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: long CPU test (minutes)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle


@pytest.fixture(autouse=True)
def _collect_cycles_after_test(request):
    """GPU tests: after each test, free what reference cycles still hold.
    A CUDA graph that a cycle keeps past its test is otherwise destroyed at the
    next garbage collection, which may fall inside another test's stream
    capture and invalidate it (graph destruction is not permitted while a
    global-mode capture is running)."""
    yield
    if request.node.get_closest_marker("gpu") is not None:
        gc.collect()
