import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libfp4q.so")
    config.addinivalue_line("markers", "slow: full-size parity case (minutes of oracle time)")


def pytest_collection_modifyitems(config, items):
    # A GPU test on a machine without a GPU is skipped, not failed, so that the
    # CPU suite can be run with or without -m "not gpu".
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
