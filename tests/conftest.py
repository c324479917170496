import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload, minutes on the GPU box")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, loaded through the binding (fails loudly if missing)."""
    import long_context_compressed_13_b300 as lc
    return lc
