import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA path)")
    config.addinivalue_line("markers", "slow: long CPU test")
    config.addinivalue_line("markers", "timeout(seconds): per-test time limit (pytest-timeout)")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
