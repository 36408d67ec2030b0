import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built libpolestar")
    config.addinivalue_line(
        "markers", "slow: large sampled parity cases at full workload sizes")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library through its C ABI (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from drift_aware_kv_spherical_gb300 import polestar
    return polestar.Library.load()
