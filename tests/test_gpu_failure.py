"""Failure detection on the GPU without a fault: a bounded wait that nobody satisfies.

The tensor-core kernels bound every mbarrier wait; when one expires the CTA records
GK_ERR_TIMEOUT in the context's device error word, frees its tensor memory and returns.
gk_selftest_wait_timeout runs that exit path with a short limit and no arriving thread. The
checks: gk_sync reports GK_ERR_TIMEOUT once (the word is cleared), the wait lasted at least
its limit and not much longer, the control case (one thread arrives) records nothing, and the
same context then runs a tensor-core product whose result matches the oracle (the tensor memory
was released and the context is still usable).
"""
import numpy as np
import pytest

import synth
from oracle import ops as oops
from tests.conftest import rel_l2

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_context_stays_usable(gkctx):
    import torch

    from gpt_decoder_gb300 import gk

    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    gk.gk_selftest_wait_timeout(gkctx, 50_000, 1, elapsed)  # control: one thread arrives
    gk.gk_sync(gkctx)
    limit = 200_000  # 200 us
    for _ in range(2):
        gk.gk_selftest_wait_timeout(gkctx, limit, 0, elapsed)
        with pytest.raises(gk.GkError) as e:
            gk.gk_sync(gkctx)
        assert e.value.status == gk.GK_ERR_TIMEOUT
        waited = int(elapsed.item())
        assert limit <= waited < limit + 50_000_000, waited
        gk.gk_sync(gkctx)  # the error word was cleared by the sync that reported it

    # a bf16 tensor-core product on the same context afterwards
    st = synth.Stream(77)
    N, K, M = 384, 256, 320
    x = st.normal(N * K).reshape(N, K).astype(np.float32)
    w = st.normal(K * M).reshape(K, M).astype(np.float32)
    xb = torch.as_tensor(x).cuda().to(torch.bfloat16)
    wb = torch.as_tensor(w).cuda().to(torch.bfloat16)
    y = torch.empty(N, M, device="cuda")
    gk.gk_matmul_fwd(gkctx, gk.GK_BF16, xb, K, wb, M, 0, None, None, 0, y, M, gk.GK_F32, N, K, M)
    gk.gk_sync(gkctx)
    ref = oops.matmul_fwd(xb.float().cpu().numpy().astype(np.float64), wb.float().cpu().numpy().astype(np.float64))
    got = y.cpu().numpy()
    assert np.abs(got - ref).max() <= 1e-4 * np.abs(ref).max()
    assert rel_l2(got, ref) < 1e-5


def test_wait_limit_is_checked_on_the_host(gkctx):
    from gpt_decoder_gb300 import gk

    for bad in (0, -5, 2_000_000_000):
        with pytest.raises(gk.GkError) as e:
            gk.gk_selftest_wait_timeout(gkctx, bad, 0)
        assert e.value.status == gk.GK_ERR_ARG
