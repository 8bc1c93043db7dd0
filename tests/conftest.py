import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libgk")
    config.addinivalue_line("markers", "slow: long-running full-size case")


def golden_values(name="page_values.txt"):
    """Parse `key = value ; source` lines of a golden fixture into a dict of floats."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split(";")[0].strip()
            if not line or line.startswith("#"):
                continue
            k, v = (s.strip() for s in line.split("="))
            out[k] = float(v)
    return out


@pytest.fixture(scope="session")
def page():
    return golden_values()
