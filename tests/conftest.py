import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 GPU and the compiled CUDA library")
    config.addinivalue_line("markers", "slow: larger CPU cases")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def cuda_lib():
    """The compiled C-ABI library; GPU tests fail loudly if it is missing."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from deterministic_top_key_gb300 import binding

    return binding.load()
