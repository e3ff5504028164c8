import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: larger CPU-only cases")


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.build()
    return o


def pytest_collection_modifyitems(config, items):
    """GPU tests need a CUDA device; elsewhere they are skipped, never faked."""
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def w12lib():
    """The CUDA library (built here if needed); no fallback exists."""
    from lossless_bit_weight_02_gb300 import _build
    _build.build()
    import lossless_bit_weight_02_gb300 as w
    w.load()
    return w
