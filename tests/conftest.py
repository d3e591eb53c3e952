import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libcsa2.so")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes of oracle time)")


def pytest_collection_modifyitems(config, items):
    # GPU tests must fail loudly, not skip, when the GPU or library is missing: the
    # product path has no CPU fallback.  Nothing to modify here; kept for clarity.
    return None
