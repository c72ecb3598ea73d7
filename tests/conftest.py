import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def pytest_collection_modifyitems(config, items):
    # GPU tests must not silently pass without a GPU: they fail loudly in the
    # fixture below instead of being skipped when -m gpu is requested.
    pass


@pytest.fixture(scope="session")
def cuda_dev():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU")
    return torch.device("cuda:0")


@pytest.fixture(scope="session")
def kvq():
    """The product binding (CUDA extension must be built)."""
    import bit_mixed_precision_kvq_gb300 as k
    k.load()  # raises if the native library is missing
    return k
