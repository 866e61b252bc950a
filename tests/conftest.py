import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    # A child run of test_oracle_pins_catch_mistakes.py: install one planted
    # mistake in the oracle before the pin modules are imported.
    plant = os.environ.get("MJ_PLANT")
    if plant:
        from tests import _plants

        _plants.apply(plant)


def load_golden(name):
    """Rows of a golden fixture under tests/golden, comments stripped."""
    path = os.path.join(ROOT, "tests", "golden", name)
    rows = []
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line)
    return rows


@pytest.fixture
def golden():
    return load_golden
