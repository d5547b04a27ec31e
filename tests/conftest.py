import os
import shutil
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libdsa.so")
    # The GPU test modules import the ctypes binding at collection time, and the binding refuses to load
    # without libdsa.so: build it (host compilation only, skipped when up to date) wherever nvcc exists.
    if shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc"):
        from compressed_sparse_attention_c4a_gb300 import build
        build.build()


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)
