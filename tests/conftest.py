import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


def _stale(lib, src):
    return not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(src)


def pytest_sessionstart(session):
    # The oracle and the input generator are plain C built with gcc; rebuild
    # them when their source is newer than the library.
    import ds4g_synth
    import oracle
    if _stale(oracle.LIBRARY, oracle.SOURCE):
        oracle.build()
    if _stale(ds4g_synth.LIBRARY, ds4g_synth.SOURCE):
        ds4g_synth.build()
    import importlib.util
    path = os.path.join(ROOT, "bit_quantized_routed_route_b300", "build.py")
    spec = importlib.util.spec_from_file_location("ds4g_build", path)
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    if b.stale():
        b.build()


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.get()
