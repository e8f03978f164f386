import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running test")


@pytest.fixture(scope="session")
def cuda():
    """The CUDA device for -m gpu tests; fails (never skips) when no GPU is visible."""
    import torch

    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import paged_kv_attention_03_gb300 as pa

    pa.build()
    pa.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pa.pa_read_device_error(clear=True, device=dev)
    return dev
