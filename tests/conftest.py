import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: full-size configuration, minutes of CPU oracle work")


def pytest_collection_modifyitems(config, items):
    # A GPU test on a machine without a GPU is a failure the user should see
    # only when they asked for GPU tests; the default CPU run deselects them
    # by marker, so nothing is skipped silently here.
    pass
