"""Test configuration: the `gpu` marker and import paths.

Tests marked `gpu` need a CUDA device and the built library; everything
else runs on the CPU (the oracle against its pins, host-side logic, the
C-ABI export table).
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device and the built CUDA library")
