"""Test configuration: the ``gpu`` marker and import paths.

``-m "not gpu"`` runs on any machine (oracle pins, host-side logic, the C ABI
symbol table); ``-m gpu`` needs a GB300 and runs the CUDA path against the
oracle.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libvnm")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def read_fixture(path):
    """Parse a ``key: value`` fixture file (``#`` starts a comment line)."""
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.strip()
    return out
