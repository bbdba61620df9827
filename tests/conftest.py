import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU and the built liblsx.so (GB300, sm_103a)")
    config.addinivalue_line(
        "markers", "slow: multi-second CPU case")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) on machines without a GPU so that
    # `pytest -m "not gpu"` and a bare `pytest` both stay green on CPU hosts.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)
