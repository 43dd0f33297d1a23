import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    # Both native pieces are built from source on whichever machine runs the
    # tests (nvcc cross-compiles here; the GPU machine builds its own).
    import oracle
    from paged_fp8_kv_quantize_gb300 import build as libbuild

    oracle.build()
    libbuild.build()


def pytest_collection_modifyitems(config, items):
    # keep file order, but make sure test_zz_* files run last
    items.sort(key=lambda it: os.path.basename(str(it.fspath)).startswith("test_zz"))
