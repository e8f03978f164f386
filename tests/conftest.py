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


def pytest_terminal_summary(terminalreporter):
    """Print the parity figures of the full-size checks (every output row of a workload
    at the size the benchmark runs) so a quiet run still shows them."""
    try:
        from _parity import RECORDS
    except Exception:
        return
    full = [(w, st) for w, st in RECORDS if w.startswith("full size")]
    if not full:
        return
    terminalreporter.write_line("parity at full size (bf16 output vs fp64 oracle; bar 1e-2 / 1e-3):")
    for w, st in full:
        terminalreporter.write_line(
            f"  {w}: {st['elems']} elems, max-abs {st['max_abs']:.2e}, mean-abs "
            f"{st['mean_abs']:.2e}; vs the bf16-rounded oracle max-abs "
            f"{st['max_abs_vs_rounded']:.2e}, mean-abs {st['mean_abs_vs_rounded']:.2e}")
