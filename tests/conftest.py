import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    # run-time specialisations compiled by the tests go to a private cache
    if "EP_GB300_JIT_CACHE" not in os.environ:
        import tempfile
        os.environ["EP_GB300_JIT_CACHE"] = tempfile.mkdtemp(prefix="ep_gb300_jit_")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run without a GPU; say so instead of failing on import.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
