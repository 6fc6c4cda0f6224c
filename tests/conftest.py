import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libvp")
    config.addinivalue_line("markers", "slow: full-size cases")


def pytest_collection_modifyitems(config, items):
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


def pytest_sessionfinish(session, exitstatus):
    """With VP_PARITY_REPORT set, writes the parity checks' error statistics there as JSON."""
    path = os.environ.get("VP_PARITY_REPORT")
    if not path:
        return
    try:
        from tests import parity
    except Exception:  # pragma: no cover
        return
    import json
    with open(path, "w") as f:
        json.dump(parity.STATS, f, indent=1, sort_keys=True)
