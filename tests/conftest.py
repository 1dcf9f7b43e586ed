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


class _KnobMonkeyPatch(pytest.MonkeyPatch):
    """pytest's monkeypatch, plus: whenever a ROWOPS_* variable is set, deleted
    or restored, the library is told to read its knobs again (it reads them
    once per process otherwise)."""

    def _reload(self):
        try:
            from row_wise_reduction_gb300 import rowops_reload_tuning

            rowops_reload_tuning()
        except Exception:  # the library is not built (some CPU-only runs): nothing to reload
            pass

    def setenv(self, name, value, prepend=None):
        super().setenv(name, value, prepend)
        if str(name).startswith("ROWOPS_"):
            self._reload()

    def delenv(self, name, raising=True):
        super().delenv(name, raising)
        if str(name).startswith("ROWOPS_"):
            self._reload()

    def undo(self):
        touched = any(str(k).startswith("ROWOPS_") for _, k, _ in getattr(self, "_setitem", []))
        super().undo()
        if touched:
            self._reload()


@pytest.fixture
def monkeypatch():
    mp = _KnobMonkeyPatch()
    yield mp
    mp.undo()
