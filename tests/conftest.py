import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU statistics test")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library, on a machine with a GPU (GPU tests fail, not skip, without one)."""
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import draft_sampling_verification_tcgen05_gb300 as dspark
    return dspark


@pytest.fixture(scope="session")
def golden_dir():
    import pathlib
    return pathlib.Path(ROOT) / "tests" / "golden"


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Totals of the GPU parity comparisons (compared positions and near-tie divergences per kind),
    printed at the end of the run and, when DSPARK_PARITY_RECORD names a file, written there."""
    from tests._helpers import PARITY_RECORD, parity_summary_lines, write_parity_record
    if not PARITY_RECORD:
        return
    for line in parity_summary_lines():
        terminalreporter.write_line(line)
    path = os.environ.get("DSPARK_PARITY_RECORD")
    if path:
        write_parity_record(path)
