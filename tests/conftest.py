import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built libzopt")


def pytest_collection_modifyitems(config, items):
    # A GPU test on a machine without CUDA is skipped rather than failed; on a GPU machine
    # the library must load (the binding raises if it is missing).
    try:
        import torch
        have_cuda = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_cuda = False
    if have_cuda:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def zopt():
    """The built library's binding (built in-tree on first use)."""
    from zero_sharded_optimizer_flat_gb300 import build_lib
    build_lib.build()
    import zero_sharded_optimizer_flat_gb300 as Z
    Z.lib()
    return Z
