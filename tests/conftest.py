import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device and the sm_103a library")
    config.addinivalue_line("markers", "slow: larger CPU oracle runs")


def _need_cpu_build():
    libs = [os.path.join(ROOT, "inputs", "libsvgen.so"), os.path.join(ROOT, "oracle", "liboracle.so")]
    srcs = [os.path.join(ROOT, "inputs", "svgen.c"), os.path.join(ROOT, "inputs", "svgen.h"),
            os.path.join(ROOT, "oracle", "oracle.c"), os.path.join(ROOT, "oracle", "oracle.h")]
    if not all(os.path.exists(p) for p in libs):
        return True
    newest_src = max(os.path.getmtime(p) for p in srcs)
    return min(os.path.getmtime(p) for p in libs) < newest_src


@pytest.fixture(scope="session", autouse=True)
def _cpu_libs():
    """The host generator and the oracle are plain C; build them if stale."""
    if _need_cpu_build():
        import __graft_entry__
        __graft_entry__.build_cpu()
    yield
