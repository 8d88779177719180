import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "large: full-size workload (tens of GB on the device)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library binding, built for sm_103a; skips without a GPU."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_recurrence_scans_gb300 as mg
    mg.load()
    return mg
