import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def gpu_lib():
    """The CUDA library, built for sm_103a; fails loudly if it cannot be loaded."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("gpu-marked test run without a CUDA device")
    import blackwell_tensor_core_02_gb300 as g

    g.load()
    return g
