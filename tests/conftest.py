import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size packs (seconds of oracle time each)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle.load()


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, loaded through the Python binding. Fails loudly when the
    library is missing: GPU tests must exercise the native path."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_pooling_gb300 as gp
    gp.load()
    return gp
