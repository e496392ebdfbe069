import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, built in-tree.  Fails loudly when it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test collected but no CUDA device is visible")
    from moe_decode_layer_gemv_gb300 import api
    return api
