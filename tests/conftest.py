import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")


@pytest.fixture(autouse=True)
def _restore_tuning():
    """Tests that force a split count or a kernel (process-wide tuning knobs
    of the library) leave every knob as they found it."""
    yield
    from helpers import restore_tuning
    restore_tuning()
