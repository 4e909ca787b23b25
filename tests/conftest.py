import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a) and the built libnomas.so")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests are only meaningful on a box with a GPU; on a CPU-only box they
    # are deselected by `-m "not gpu"`.  When selected without a GPU they fail
    # loudly (no silent skip) so a missing device cannot pass as green.
    pass
