import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 (sm_103) GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    """GPU tests fail loudly (rather than skip) when no GPU is present, except
    when they were deselected with -m 'not gpu'."""
    return None
