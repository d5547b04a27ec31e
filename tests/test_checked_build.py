"""The bounds-checked build: libdsa_checked.so compiles the same kernels with -DDSA_CHECKED, which bounds-checks
their computed shared-memory and table indexes (a bad index records DSA_ERR_DEVICE_FAULT and the access is
skipped, never a trap).  It exports the same entry points, the binding loads it under DSA_CHECKED=1, and the
stage parity cases pass through it with a zero device status."""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def checked_lib():
    from compressed_sparse_attention_c4a_gb300 import build
    return build.build(checked=True)


def test_checked_build_exports_every_entry_point(checked_lib):
    from test_abi import _declared
    lib = ctypes.CDLL(checked_lib)
    for n in _declared():
        assert hasattr(lib, n), n
    env = dict(os.environ, DSA_CHECKED="1")
    out = subprocess.run([sys.executable, "-c", "from compressed_sparse_attention_c4a_gb300 import dsa; print(dsa._PATH)"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    assert out.stdout.strip().endswith("libdsa_checked.so")


@pytest.mark.gpu
def test_checked_build_passes_the_stage_parity_cases(checked_lib):
    env = dict(os.environ, DSA_CHECKED="1")
    sel = ("test_compress_main_and_swa or test_compress_indexer or test_index_scores or test_topk or "
           "test_attention or test_index_unmapped_block or test_attention_unmapped_block")
    res = subprocess.run([sys.executable, "-m", "pytest", os.path.join("tests", "test_gpu_stages.py"), "-m", "gpu", "-q",
                          "-x", "-p", "no:cacheprovider", "-k", sel], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=1200)
    assert res.returncode == 0, res.stdout[-4000:] + res.stderr[-2000:]
    assert " passed" in res.stdout and " failed" not in res.stdout
