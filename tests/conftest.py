import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def _have_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _have_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this process")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session", autouse=True)
def _short_kernel_watchdog():
    """On a GPU, give every pipeline wait 250 ms (legitimate waits take
    microseconds), so a stalled kernel fails its test quickly instead of
    holding the GPU for the default 2 s per wait."""
    if not _have_gpu():
        yield
        return
    from exact_io_aware_12_gb300 import _lib
    _lib.fa_set_wait_limit_ns(250_000_000)
    yield
    _lib.fa_set_wait_limit_ns(0)
