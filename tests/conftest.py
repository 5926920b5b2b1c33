import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line(
        "markers", "slow: full-size CPU work (minutes)")


import pytest  # noqa: E402


def _lib_stale(lib, srcs):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in srcs)


@pytest.fixture(scope="session")
def mpk_lib():
    """The compiled C-ABI library, (re)built in-tree when missing or older
    than its sources."""
    import glob
    from task_graph_runtime_gb300 import build, mpk
    srcs = glob.glob(os.path.join(ROOT, "task_graph_runtime_gb300", "csrc",
                                  "*")) + [os.path.join(ROOT, "include",
                                                        "mpk.h")]
    if _lib_stale(mpk.LIB_PATH, srcs):
        build.build()
    return mpk.load_library()
