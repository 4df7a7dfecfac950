import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


@pytest.fixture(scope="session")
def cuda_device():
    """The CUDA device the gpu-marked tests run on.  A GPU test that finds no
    GPU fails instead of skipping: a silent skip would hide a missing path."""
    import torch
    assert torch.cuda.is_available(), "gpu-marked test run without a CUDA device"
    return torch.device("cuda", 0)


@pytest.fixture(scope="session")
def fp8lin(cuda_device):
    """The product binding (builds the library when it is missing)."""
    import __graft_entry__
    __graft_entry__._build_module().build()
    import float8_linear_layers_gb300 as m
    return m
