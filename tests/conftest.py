import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    # Build libtw.so (nvcc cross-compiles for sm_103a without a GPU) and the oracle
    # if they are missing or older than their sources.
    import __graft_entry__
    __graft_entry__._build_module().build()
    import oracle
    oracle.build()
    oracle.build(openmp=True)


def pytest_collection_modifyitems(config, items):
    # A gpu-marked test on a machine without a GPU is skipped, never silently rerouted.
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
