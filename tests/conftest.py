import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # keep the file order stable: pytest collects files alphabetically
    pass


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library, loaded through the Python binding."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from io_aware_exact_attn_gb300 import _ffi
    return _ffi.lib()
