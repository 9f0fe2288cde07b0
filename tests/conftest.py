import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library through its Python binding (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from int4_weight_only_w4a16_gb300 import binding
    return binding


@pytest.fixture(scope="session")
def host_lib():
    """The library built and loaded for host-only entry points (no GPU needed)."""
    from int4_weight_only_w4a16_gb300 import binding, build
    build.build()
    binding.load()
    return binding
