import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_sessionstart(session):
    """Build libmsa.so and the C oracle if they are missing or older than
    their sources (incremental: nothing to do when up to date), so that the
    suite runs on a fresh checkout."""
    from kv_cache_segment_gb300 import build
    build.build()
    import oracle
    oracle.build_oracle()
