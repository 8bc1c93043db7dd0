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


def assert_close(got, ref, tol, what=""):
    """Parity of a GPU output with its reference: EVERY element within tol * max|ref| (a wrong
    tile, edge, row or column fails this even where a norm over millions of elements would not),
    and the relative L2 of the whole below tol."""
    import numpy as np

    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    if got.size == 0:
        return
    err = np.abs(got - ref)
    scale = max(float(np.abs(ref).max()), 1e-30)
    worst = float(err.max())
    if not worst <= tol * scale:
        at = np.unravel_index(int(np.nanargmax(err)), err.shape)
        raise AssertionError(f"{what}: max |err| {worst:.3e} at {at} exceeds {tol} x max|ref| {scale:.3e}")
    r = rel_l2(got, ref)
    assert r < tol, f"{what}: relative L2 {r:.3e} >= {tol}"


@pytest.fixture(autouse=True)
def _float32_default_dtype():
    """GPU buffers are allocated with torch's default dtype: keep it float32 for every test."""
    import torch

    torch.set_default_dtype(torch.float32)
    yield
