import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(autouse=True)
def _reset_oracle_mutant():
    """Every test starts and ends with the correct oracle (mutant 0)."""
    yield
    if "oracle" in sys.modules:
        sys.modules["oracle"].set_mutant(0)
