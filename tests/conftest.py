import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 (sm_103) GPU and the CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.lib()  # builds the C oracle if needed
    return oracle


@pytest.fixture(scope="session")
def fp8bs():
    """The CUDA library's Python binding, on a GPU machine only."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import fp8_fine_grained_18_b300 as lib
    return lib
