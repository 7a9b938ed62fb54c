import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def ensure_lib():
    """Build libvg.so in-tree if it is not there (nvcc cross-compiles without a GPU)."""
    lib = os.path.join(ROOT, "self_speculative_sparse_vg_gb300", "libvg.so")
    if not os.path.exists(lib):
        from self_speculative_sparse_vg_gb300 import build
        build.build()
