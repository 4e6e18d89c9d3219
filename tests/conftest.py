import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _lib_is_stale():
    from paged_kv_gqa_rope_gb300 import build
    if not os.path.exists(build.LIB):
        return True
    t = os.path.getmtime(build.LIB)
    deps = build.sources() + [os.path.join(build.CSRC, f) for f in os.listdir(build.CSRC)] + \
        [os.path.join(build.INCLUDE, f) for f in os.listdir(build.INCLUDE)]
    return any(os.path.getmtime(p) > t for p in deps)


@pytest.fixture(scope="session")
def libpa():
    """libpa.so, built in-tree first if it is missing or older than its sources."""
    from paged_kv_gqa_rope_gb300 import build, pa
    if _lib_is_stale():
        build.build()
    return pa.lib()
