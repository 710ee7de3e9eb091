"""Shared pytest configuration.

Tests marked ``gpu`` need a CUDA device (they run the library's kernels); every
other test runs on a CPU-only host."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")
