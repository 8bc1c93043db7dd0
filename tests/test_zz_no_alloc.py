"""gk_layernorm_bwd_noalloc, the LayerNorm backward for callers that cannot allocate device
memory, against the context-based gk_layernorm_bwd on the same inputs.

Its scratch is a fixed array inside the library that keeps the previous call's contents, so
the check makes two calls in a row, of different shapes, and compares each with the
workspace-based entry point. This file sorts last so that a run stopping at the first failure
has run everything else first; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

import synth
from tests.conftest import rel_l2

pytestmark = pytest.mark.gpu


def _case(seed, rows, C):
    st = synth.Stream(seed)
    x = st.normal(rows * C).reshape(rows, C) * 2 + 0.5
    gm, bt = st.normal(C), st.normal(C)
    g = st.normal(rows * C).reshape(rows, C)
    mu = x.astype(np.float64).mean(1)
    rs = 1.0 / np.sqrt(((x - mu[:, None]) ** 2).mean(1) + 1e-5)
    dx0 = st.normal(rows * C).reshape(rows, C)
    dg0, db0 = st.normal(C), st.normal(C)
    return x, gm, g, mu.astype(np.float32), rs.astype(np.float32), dx0, dg0, db0


def _run(fn, args, torch, rows, C, acc):
    x, gm, g, mu, rs, dx0, dg0, db0 = args
    d = lambda a: torch.as_tensor(np.ascontiguousarray(a)).cuda()
    dx, dgm, dbt = d(dx0), d(dg0), d(db0)
    dxb = torch.empty(rows, C, dtype=torch.bfloat16, device="cuda")
    fn(d(x), d(gm), d(mu), d(rs), d(g), dx, acc, dxb, dgm, dbt)
    torch.cuda.synchronize()
    return dx.cpu().numpy(), dxb.float().cpu().numpy(), dgm.cpu().numpy(), dbt.cpu().numpy()


@pytest.mark.parametrize("order", [((4096, 768, 1), (37, 96, 0)), ((5, 130, 0), (4096, 768, 1))])
def test_noalloc_matches_workspace_entry_point_twice(gkctx, order):
    import torch

    from gpt_decoder_gb300 import gk

    stream = torch.cuda.current_stream()
    for i, (rows, C, acc) in enumerate(order):
        args = _case(1000 + 17 * i + C, rows, C)

        def ref_fn(x, gm, mu, rs, g, dx, a, dxb, dgm, dbt):
            gk.gk_layernorm_bwd(gkctx, x, gm, mu, rs, g, dx, a, dxb, dgm, dbt, rows, C)
            gk.gk_sync(gkctx)

        def na_fn(x, gm, mu, rs, g, dx, a, dxb, dgm, dbt):
            gk.gk_layernorm_bwd_noalloc(stream, x, gm, mu, rs, g, dx, a, dxb, dgm, dbt, rows, C)

        want = _run(ref_fn, args, torch, rows, C, acc)
        got = _run(na_fn, args, torch, rows, C, acc)
        # dx and its bf16 copy are per-row results: identical; dgamma / dbeta may group rows
        # into partial sums differently, so they get the LayerNorm tests' tolerance
        assert np.array_equal(got[0], want[0])
        assert np.array_equal(got[1], want[1])
        assert rel_l2(got[2], want[2]) < 1e-5
        assert rel_l2(got[3], want[3]) < 1e-5


def test_noalloc_rejects_rows_wider_than_its_scratch(gkctx):
    import torch

    from gpt_decoder_gb300 import gk

    z = torch.zeros(4, device="cuda")
    with pytest.raises(gk.GkError) as e:
        gk.gk_layernorm_bwd_noalloc(0, z, z, z, z, z, z, 0, None, z, z, 1, 524289)
    assert e.value.status == gk.GK_ERR_WORKSPACE
    with pytest.raises(gk.GkError) as e:
        gk.gk_layernorm_bwd_noalloc(0, None, z, z, z, z, z, 0, None, z, z, 1, 4)
    assert e.value.status == gk.GK_ERR_ARG
