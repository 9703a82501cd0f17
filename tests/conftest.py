import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload checks")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def cblib():
    """The product C-ABI library (built on demand); host-side calls only."""
    from conv_bn_activation_gb300 import _build, binding
    _build.build_library()
    return binding


@pytest.fixture(scope="session")
def gpu():
    """A CUDA device and the built library; skips nothing -- gpu tests must run on a GPU."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test selected but no CUDA device is visible")
    from conv_bn_activation_gb300 import _build, binding
    _build.build_library()
    binding.load()
    return torch.device("cuda:0")
