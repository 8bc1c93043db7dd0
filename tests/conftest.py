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


@pytest.fixture(scope="session")
def gkctx():
    """A libgk context on the current torch stream (GPU tests only)."""
    import torch

    from gpt_decoder_gb300 import gk

    ctx = gk.Ctx(torch.cuda.current_stream().cuda_stream, workspace_bytes=256 << 20)
    yield ctx
    ctx.close()


def rel_l2(a, b):
    import numpy as np

    a = np.asarray(a, dtype=np.float64).ravel()
    b = np.asarray(b, dtype=np.float64).ravel()
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


@pytest.fixture(autouse=True)
def _float32_default_dtype():
    """GPU buffers are allocated with torch's default dtype: keep it float32 for every test."""
    import torch

    torch.set_default_dtype(torch.float32)
    yield
