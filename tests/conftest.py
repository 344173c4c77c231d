"""pytest configuration: the ``gpu`` marker and shared fixtures."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device on this host")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


class _Opts:
    """la_debug_set's test switches (the library's process-wide options)."""

    def __init__(self, la):
        self.la = la

    def path(self, name: str):
        """'auto', 'simt' (the fp32 CUDA-core kernels) or 'tc' (the tensor cores)."""
        self.la.debug_set(self.la.LA_OPT_PATH, {"auto": 0, "simt": 1, "tc": 2}[name])

    def lockstep(self, on: bool = True):
        self.la.debug_set(self.la.LA_OPT_TC_LOCKSTEP, int(on))

    def force_timeout(self, on: bool = True):
        self.la.debug_set(self.la.LA_OPT_FORCE_TIMEOUT, int(on))

    def reset(self):
        for o in (self.la.LA_OPT_PATH, self.la.LA_OPT_TC_LOCKSTEP, self.la.LA_OPT_FORCE_TIMEOUT):
            self.la.debug_set(o, 0)


@pytest.fixture
def opts():
    """Set the library's test switches; every switch is back to 0 after the test."""
    import retnet_retention_gb300 as la
    o = _Opts(la)
    o.reset()
    yield o
    o.reset()
