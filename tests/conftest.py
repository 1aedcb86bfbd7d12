import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300) and the built libcbs.so")
    config.addinivalue_line("markers", "slow: long-running CPU check")


@pytest.fixture(scope="session")
def cuda_lib():
    """Build (if needed) and load libcbs.so; skip nothing: GPU tests need it."""
    from conv_bn_silu_gb300 import build
    build.build()
    from conv_bn_silu_gb300 import _binding
    return _binding.lib()
