import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")
    config.addinivalue_line("markers", "slow: long-running CPU check")


@pytest.fixture(scope="session")
def cuda_dev():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device (select CPU tests with -m 'not gpu')")
    return torch.device("cuda:0")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """The parity checks of the run with the largest max-abs error against the tensor's RMS (the
    literal reading of the bound), beside the per-row reading the tests assert."""
    try:
        from parity import MAX_ABS_RMS, RECORDS
    except Exception:
        return
    if not RECORDS:
        return
    tr = terminalreporter
    tr.section("parity: max-abs error against RMS")
    over = sum(1 for r in RECORDS if r[3] > MAX_ABS_RMS)
    tr.write_line(f"{len(RECORDS)} checks; worst rel-Frobenius {max(r[1] for r in RECORDS):.2e}, worst per-row "
                  f"max-abs/RMS {max(r[2] for r in RECORDS):.2e}; {over} above {MAX_ABS_RMS:g} x RMS(tensor)")
    for what, rel, mx, gl in sorted(RECORDS, key=lambda r: -r[3])[:12]:
        tr.write_line(f"  {gl:9.2e} tensor  {mx:9.2e} row  {rel:9.2e} fro   {what}")
