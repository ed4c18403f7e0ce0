import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


def _has_gpu() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.hookimpl(hookwrapper=True)
def pytest_runtest_call(item):
    """Each GPU test runs inside an NVTX range named after it, so that a profiler's range
    filter (ncu --nvtx --nvtx-include) can pick one test's products out of a session."""
    nvtx = None
    if "gpu" in item.keywords and _has_gpu():
        import torch
        nvtx = torch.cuda.nvtx
        nvtx.range_push(item.nodeid)
    try:
        yield
    finally:
        if nvtx is not None:
            nvtx.range_pop()
