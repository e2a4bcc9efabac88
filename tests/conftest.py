import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload")


@pytest.fixture(scope="session")
def cuda():
    """The CUDA library; on a GPU machine a missing build is an error, not a skip."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_recurrence_scan_chunked_gb300 as lrs
    lrs.load()  # raises if the shared library is missing
    return lrs
