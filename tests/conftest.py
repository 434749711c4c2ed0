import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def printed():
    with open(os.path.join(ROOT, "tests", "golden", "printed_values.json")) as f:
        return json.load(f)


def has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


def pytest_terminal_summary(terminalreporter):
    """Repeat the parity figures the GPU tests printed (raw max|err|/rms of every
    bf16 comparison, stage-by-stage agreement) at the end of the run."""
    from tests import parity_log
    if parity_log.LINES:
        terminalreporter.section("parity figures")
        for line in parity_log.LINES:
            terminalreporter.write_line(line)
