"""Pins of the oracle's generic ops (Add with broadcast, Mul, Scale, Sum, Tanh, SGD) and of its
two small-network trainers, against torch autograd in float64, finite differences, closed
forms, the scalar reverse-mode engine, and what the pages say their runs do."""
import random

import numpy as np
import pytest

import synth
from oracle import mlp, ops
from oracle.scalar_ad import Var, vsum


def _t():
    return pytest.importorskip("torch")


def _rand(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def test_generic_ops_match_torch_autograd():
    torch = _t()
    a, b, bias, g = _rand(1, 5, 7), _rand(2, 5, 7), _rand(3, 7), _rand(4, 5, 7)
    ta, tb, tbias = (torch.tensor(x, requires_grad=True) for x in (a, b, bias))
    tg = torch.tensor(g)
    cases = [
        ("add", lambda: ta + tbias, ops.add_fwd(a, bias), ops.add_bwd(g, bias.shape), (ta, tbias)),
        ("mul", lambda: ta * tb, ops.mul_fwd(a, b), ops.mul_bwd(a, b, g), (ta, tb)),
        ("scale", lambda: -0.37 * ta, ops.scale_fwd(a, -0.37), (ops.scale_bwd(-0.37, g),), (ta,)),
        ("tanh", lambda: torch.tanh(ta), ops.tanh_fwd(a), (ops.tanh_bwd(np.tanh(a), g),), (ta,)),
    ]
    for name, f, fwd, grads, inputs in cases:
        for t in inputs:
            t.grad = None
        y = f()
        np.testing.assert_allclose(fwd, y.detach().numpy(), rtol=1e-13, atol=1e-13, err_msg=name)
        y.backward(tg)
        for got, t in zip(grads, inputs):
            np.testing.assert_allclose(got, t.grad.numpy(), rtol=1e-13, atol=1e-13, err_msg=name)
    ta.grad = None
    s = ta.sum()
    assert ops.sum_fwd(a) == pytest.approx(s.item(), rel=1e-14)
    s.backward(torch.tensor(2.5, dtype=torch.float64))
    np.testing.assert_array_equal(ops.sum_bwd(a.shape, 2.5), ta.grad.numpy())


def test_generic_ops_closed_forms_and_finite_differences():
    # tanh(0) = 0, tanh'(0) = 1; tanh' = 1 - tanh^2 by central differences
    assert ops.tanh_fwd(0.0) == 0.0 and ops.tanh_bwd(0.0, 1.0) == 1.0
    x = np.linspace(-3, 3, 13)
    h = 1e-6
    np.testing.assert_allclose(ops.tanh_bwd(np.tanh(x), 1.0), (np.tanh(x + h) - np.tanh(x - h)) / (2 * h),
                               rtol=1e-8, atol=1e-9)
    # the broadcast bias gradient is the column sum; Sum of ones counts the elements
    g = np.arange(12.0).reshape(3, 4)
    np.testing.assert_array_equal(ops.add_bwd(g, (4,))[1], [12, 15, 18, 21])
    assert ops.sum_fwd(np.ones((6, 7))) == 42
    # Mul by ones is the identity, and its gradient on the other side is g itself
    np.testing.assert_array_equal(ops.mul_bwd(np.ones(3), np.array([1.0, 2, 3]), np.ones(3))[1], np.ones(3))
    np.testing.assert_array_equal(ops.sgd(np.array([1.0, 2.0]), np.array([10.0, -10.0]), 0.05), [0.5, 2.5])


def _torch_circle(xs, ys, params, opt, steps):
    torch = _t()
    p = [torch.tensor(np.asarray(t, np.float64), requires_grad=True) for t in params]
    o = (torch.optim.SGD(p, lr=0.05) if opt == "sgd"
         else torch.optim.AdamW(p, lr=0.05, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0))
    x = torch.tensor(xs, dtype=torch.float64)
    y = torch.tensor(ys, dtype=torch.long)
    losses = []
    for _ in range(steps + 1):
        logits = torch.tanh(x @ p[0] + p[1]) @ p[2] + p[3]
        loss = torch.nn.functional.cross_entropy(logits, y)
        losses.append(loss.item())
        o.zero_grad()
        loss.backward()
        o.step()
    return np.array(losses)


@pytest.mark.parametrize("opt", ["sgd", "adamw"])
def test_circle_trainer_matches_torch(opt):
    xs, ys, params = synth.circle_case(3)
    got, _, _ = mlp.train_circle(xs, ys, *params, opt=opt, steps=40)
    np.testing.assert_allclose(got, _torch_circle(xs, ys, params, opt, 40), rtol=1e-10, atol=1e-12)


def test_circle_trainer_behaves_as_the_pages_report():
    # [LM1] "Training loop": with lr 0.05 SGD creeps (loss falling slowly, accuracy rising)
    # while AdamW solves the task (near-zero loss, 100% accuracy by step 100-200)
    xs, ys, params = synth.circle_case(3)
    ls, acc_s, _ = mlp.train_circle(xs, ys, *params, opt="sgd")
    la, acc_a, _ = mlp.train_circle(xs, ys, *params, opt="adamw")
    ck = list(range(0, 501, 100))
    assert all(ls[i] > ls[j] for i, j in zip(ck, ck[1:]))
    assert acc_s[500] > acc_s[0] and ls[500] > 0.3
    assert la[100] < 0.15 and acc_a[200] >= 0.99 and la[500] < 0.03


def test_xor_trainer_equals_the_scalar_engine():
    """The tensor-op XOR trainer against the scalar reverse-mode engine ([AD] Step 5's
    micrograd network) from the same initial weights: the same loss at every step."""
    rng = random.Random(42)
    neurons1 = [[rng.uniform(-1, 1) for _ in range(2)] for _ in range(4)]
    neurons2 = [[rng.uniform(-1, 1) for _ in range(4)]]
    w1, w2 = np.array(neurons1).T, np.array(neurons2).T  # [in, out]
    xs = np.array([[0, 0], [0, 1], [1, 0], [1, 1]], float)
    ys = np.array([[-1], [1], [1], [-1]], float)
    got, _ = mlp.train_xor(xs, ys, w1, np.zeros(4), w2, np.zeros(1), steps=60)

    layers = [[([Var(w) for w in ws], Var(0.0)) for ws in neurons] for neurons in (neurons1, neurons2)]
    params = [p for layer in layers for (ws, b) in layer for p in ws + [b]]

    def model(x):
        for layer in layers:
            x = [vsum([wi * xi for wi, xi in zip(ws, x)] + [b]).tanh() for ws, b in layer]
        return x[0]

    ref = []
    for _ in range(60):
        loss = vsum([(model(x) - y) ** 2 for x, y in zip(xs.tolist(), ys.ravel().tolist())])
        for p in params:
            p.grad = 0.0
        loss.backward()
        for p in params:
            p.value -= 0.05 * p.grad
        ref.append(loss.value)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_xor_trainer_learns():
    xs, ys, params = synth.xor_case(5)
    losses, pred = mlp.train_xor(xs, ys, *params, steps=100)
    assert losses[-1] < losses[0]
    losses, pred = mlp.train_xor(xs, ys, *params, steps=1000)
    assert (np.sign(pred) == ys).all() and losses[-1] < 0.1
