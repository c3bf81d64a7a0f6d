import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU")


def pytest_sessionstart(session):
    """Build libpagedkv.so (nvcc cross-compiles for sm_103a, no GPU needed)
    when it is missing or older than its sources, so a fresh checkout tests
    the library it holds.  The package itself never builds or falls back:
    loading a missing library raises."""
    from paged_kv_cache_162_gb300 import _build
    if not _build.up_to_date():
        _build.build()


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
