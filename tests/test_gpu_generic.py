"""Generic ops (Add with broadcast, Mul, Scale, Sum, Tanh), SGD and the pages' two small
networks on the GPU against the oracle."""
import numpy as np
import pytest

import synth
from oracle import mlp as omlp
from oracle import ops

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch

    return torch.as_tensor(np.ascontiguousarray(a, np.float32)).cuda()


def _host(t):
    return t.cpu().numpy().astype(np.float64)


def _normal(seed, *shape):
    return synth.Stream(seed).normal(int(np.prod(shape))).reshape(shape)


# (rows, m): b has m elements broadcast over rows (rows = 1: the plain elementwise sum)
SIZES = [(1, 1), (1, 7), (1000, 37), (4096, 768), (1, 3 * 1024 + 5), (3, 100_003)]


@pytest.mark.parametrize("rows,m", SIZES)
@pytest.mark.parametrize("acc", [0, 1])
def test_add_fwd_bwd(gkctx, rows, m, acc):
    from gpt_decoder_gb300 import gk

    n = rows * m
    a, b, g = _normal(1 + n, n), _normal(2 + n, m), _normal(3 + n, n)
    prior_a, prior_b = _normal(4 + n, n), _normal(5 + n, m)
    y = _dev(np.zeros(n))
    gk.gk_add_fwd(gkctx, _dev(a), _dev(b), y, n, m)
    da, db = _dev(prior_a), _dev(prior_b)
    gk.gk_add_bwd(gkctx, _dev(g), da, db, n, m, acc)
    gk.gk_sync(gkctx)
    ref = ops.add_fwd(a.reshape(-1, m), b).reshape(-1)
    rda, rdb = ops.add_bwd(g.reshape(-1, m), (m,))
    np.testing.assert_allclose(_host(y), ref, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(_host(da), rda.reshape(-1) + (prior_a if acc else 0), rtol=1e-6, atol=1e-6)
    # the bias gradient is a float32 rounding of the float64 column sums
    np.testing.assert_allclose(_host(db), rdb + (prior_b if acc else 0), rtol=1e-6, atol=1e-6 * np.sqrt(n // m))


@pytest.mark.parametrize("n", [1, 5, 1 << 20, (1 << 22) + 3])
@pytest.mark.parametrize("acc", [0, 1])
def test_mul_scale_tanh(gkctx, n, acc):
    from gpt_decoder_gb300 import gk

    a, b, g, prior = _normal(11, n), _normal(12, n), _normal(13, n), _normal(14, n)
    base = prior if acc else 0
    y, da, db = _dev(np.zeros(n)), _dev(prior), _dev(prior)
    gk.gk_mul_fwd(gkctx, _dev(a), _dev(b), y, n)
    gk.gk_mul_bwd(gkctx, _dev(g), _dev(a), _dev(b), da, db, n, acc)
    gk.gk_sync(gkctx)
    rda, rdb = ops.mul_bwd(a, b, g)
    np.testing.assert_allclose(_host(y), ops.mul_fwd(a, b), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(_host(da), rda + base, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(_host(db), rdb + base, rtol=1e-6, atol=1e-6)

    ys, ds = _dev(np.zeros(n)), _dev(prior)
    gk.gk_scale_fwd(gkctx, _dev(a), -0.37, ys, n)
    gk.gk_scale_bwd(gkctx, _dev(g), -0.37, ds, n, acc)
    yt, dt = _dev(np.zeros(n)), _dev(prior)
    gk.gk_tanh_fwd(gkctx, _dev(a), yt, n)
    gk.gk_tanh_bwd(gkctx, yt, _dev(g), dt, n, acc)
    gk.gk_sync(gkctx)
    np.testing.assert_allclose(_host(ys), ops.scale_fwd(a, -0.37), rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(_host(ds), ops.scale_bwd(-0.37, g) + base, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(_host(yt), ops.tanh_fwd(a), rtol=2e-6, atol=2e-7)
    np.testing.assert_allclose(_host(dt), ops.tanh_bwd(ops.tanh_fwd(a), g) + base, rtol=1e-5, atol=1e-6)


def test_elementwise_in_place(gkctx):
    from gpt_decoder_gb300 import gk

    n = 1001
    a, b = _normal(21, n), _normal(22, n)
    t = _dev(a)
    gk.gk_add_fwd(gkctx, t, _dev(b), t, n, n)
    gk.gk_tanh_fwd(gkctx, t, t, n)
    gk.gk_scale_fwd(gkctx, t, 2.0, t, n)
    gk.gk_sync(gkctx)
    np.testing.assert_allclose(_host(t), 2.0 * np.tanh(a + b), rtol=2e-6, atol=2e-7)


@pytest.mark.parametrize("n", [0, 1, 255, 1 << 20, 50_000_003])
def test_sum_fwd_bwd(gkctx, n):
    import torch

    from gpt_decoder_gb300 import gk

    a = _normal(31, n) if n else np.zeros(0, np.float32)
    y = torch.full((1,), 7.0, device="cuda")
    gk.gk_sum_fwd(gkctx, _dev(a) if n else None, y, n)
    gk.gk_sync(gkctx)
    assert abs(float(y.item()) - ops.sum_fwd(a)) <= 1e-6 * max(1.0, np.abs(a).sum())
    if n:
        da = _dev(np.ones(n))
        gk.gk_sum_bwd(gkctx, _dev(np.array([0.25])), da, n, 1)
        gk.gk_sync(gkctx)
        np.testing.assert_array_equal(_host(da)[:1000], np.full(min(n, 1000), 1.25))


def test_sgd_step(gkctx):
    from gpt_decoder_gb300 import gk

    n = 12345
    p, g = _normal(41, n), _normal(42, n)
    t = _dev(p)
    gk.gk_sgd_step(gkctx, t, _dev(g), n, 0.05)
    gk.gk_sync(gkctx)
    np.testing.assert_allclose(_host(t), ops.sgd(p, g, 0.05), rtol=1e-6, atol=1e-7)


def test_generic_ops_reject_bad_arguments(gkctx):
    from gpt_decoder_gb300 import gk

    t = _dev(np.zeros(12))
    with pytest.raises(gk.GkError) as e:
        gk.gk_add_fwd(gkctx, t, t, t, 12, 5)  # 5 does not divide 12
    assert e.value.status == gk.GK_ERR_ARG
    with pytest.raises(gk.GkError) as e:
        gk.gk_mul_fwd(gkctx, t, None, t, 12)
    assert e.value.status == gk.GK_ERR_ARG
    gk.gk_mul_fwd(gkctx, None, None, None, 0)  # empty: nothing to do


@pytest.mark.parametrize("opt", ["sgd", "adamw"])
def test_circle_network_trains_like_the_oracle(gkctx, opt):
    """[LM1] "Training loop": the 2 -> 16 -> 2 tanh network on the circle task, 501 iterations,
    float32 on the GPU against the float64 oracle."""
    from gpt_decoder_gb300 import mlp

    xs, ys, params = synth.circle_case(3)
    got_l, got_a, got_p = mlp.train_circle(gkctx, xs, ys, *params, opt=opt)
    ref_l, ref_a, ref_p = omlp.train_circle(xs, ys, *params, opt=opt)
    np.testing.assert_allclose(got_l, ref_l, rtol=2e-4, atol=2e-5)
    assert np.abs(got_a - ref_a).max() <= 2 / 256  # a point or two on the boundary
    for g, r in zip(got_p, ref_p):
        np.testing.assert_allclose(g, r, rtol=2e-3, atol=2e-4)


def test_xor_network_trains_like_the_oracle(gkctx):
    """[AD] Step 5: the [2, 4, 1] tanh network on XOR, sum of squares, SGD; every op of the
    generic set (Add, Scale, Mul, Sum, Tanh) is on the path."""
    from gpt_decoder_gb300 import mlp

    xs, ys, params = synth.xor_case(5)
    got_l, got_pred = mlp.train_xor(gkctx, xs, ys, *params, steps=300)
    ref_l, ref_pred = omlp.train_xor(xs, ys, *params, steps=300)
    np.testing.assert_allclose(got_l, ref_l, rtol=1e-4, atol=1e-6)
    np.testing.assert_allclose(got_pred, ref_pred, rtol=1e-4, atol=1e-5)
    assert (np.sign(got_pred) == ys).all()
