import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.dirname(os.path.abspath(__file__))):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library's Python binding; the test fails (not skips) if the
    extension cannot be loaded on a GPU machine."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import token_tree_verification_gb300 as ttv
    lib = ttv.load()
    # SPEC_TREE_CHECKED=1 runs the suites against the bounds-checked build
    want = 1 if os.environ.get("SPEC_TREE_CHECKED", "0") == "1" else 0
    assert lib.spec_build_checked() == want, ttv.lib_path()
    return ttv
