import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity cases (minutes)")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when CUDA is missing: the product path
    # has no CPU fallback, so a GPU run without a GPU is an error.
    pass
