"""Shared test set-up: the ``gpu`` marker, import paths and the oracle build."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); parity tests through the C ABI")


@pytest.fixture(scope="session")
def oracle():
    from oracle import oracle as _oracle

    _oracle.build()
    return _oracle
