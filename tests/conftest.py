import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def dev():
    """The CUDA device for GPU tests; the product library is loaded up front so
    a missing extension fails loudly instead of skipping."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a CUDA device")
    import nvfp4_speculative_draft_gb300 as nd
    nd.load()
    return torch.device("cuda:0")
