import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libliger.so")
    config.addinivalue_line("markers", "slow: long-running case")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library on a CUDA device; builds it if needed."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_rmsnorm_fwd_gb300 import _native
    _native.load()
    return _native
