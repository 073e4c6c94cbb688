"""Shared pytest setup: the ``gpu`` marker and import paths.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything else runs on
a CPU-only machine (oracle pins, host-side argument checks, the library's symbol table).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled libtv.so")


@pytest.fixture(scope="session")
def tvlib():
    """The product binding, built if needed (compiles on CPU; calls need a GPU)."""
    from speculative_decoding_tree_04_gb300 import build as tvbuild
    tvbuild.build()
    from speculative_decoding_tree_04_gb300 import tv
    return tv
