import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU check")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.lib()


def pytest_collection_modifyitems(config, items):
    """GPU tests skip (not fail) on a machine without CUDA; on a GPU machine they run
    against the built library and fail loudly if it cannot be built or loaded."""
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
def kdlib():
    """The built CUDA library (built on first use)."""
    from session_decode_step_gb300 import build
    import session_decode_step_gb300 as kd
    build.build()
    kd.lib()
    return kd
