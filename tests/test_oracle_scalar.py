"""Pins of the oracle's scalar reverse-mode engine against the worked examples the pages print."""
import math
import random

import numpy as np
import pytest

from oracle.scalar_ad import Dual, Var, dual_derivative, vsum


def test_tiny_graph(page):
    # L = (w x + b)^2 with z used twice: gradients of the two uses add up.
    w, x, b = Var(2), Var(3), Var(1)
    z = w * x + b
    L = z * z
    L.backward()
    assert z.value == page["tiny_graph.z"] and L.value == page["tiny_graph.L"]
    assert z.grad == page["tiny_graph.dL_dz"]
    assert w.grad == page["tiny_graph.dL_dw"]
    assert x.grad == page["tiny_graph.dL_dx"]
    assert b.grad == page["tiny_graph.dL_db"]


class _AssigningMul(Var):
    """A deliberately wrong engine: backward assigns (=) instead of adding (+=)."""

    def backward(self):
        seen, stack, nodes = set(), [self], []
        while stack:
            n = stack.pop()
            if id(n) in seen:
                continue
            seen.add(id(n))
            nodes.append(n)
            stack.extend(p for p, _ in n.parents)
        nodes.sort(key=lambda n: n.serial, reverse=True)
        self.grad = 1.0
        for n in nodes:
            for p, d in n.parents:
                p.grad = d * n.grad  # the mutation


def _fd(f, x, h):
    return (f(x + h) - f(x - h)) / (2 * h)


def _rel(a, n):
    return abs(a - n) / (abs(a) + abs(n))


def test_plus_equals_and_its_mutation(page):
    z = Var(7)
    L = z * z
    L.backward()
    assert z.grad == page["mul_twice.dL_dz"]
    num = _fd(lambda t: t * t, 7.0, page["gradcheck.h"])
    assert _rel(z.grad, num) < page["gradcheck.threshold"]
    # Planting the "=" mistake halves the gradient and the gradient check catches it.
    z2 = Var(7)
    L2 = _AssigningMul(z2.value * z2.value, ((z2, z2.value), (z2, z2.value)))
    L2.backward()
    assert z2.grad == page["mul_assign.dL_dz"]
    assert _rel(z2.grad, num) > page["gradcheck.threshold"]


def test_sin_of_square_reverse_and_forward(page):
    x = Var(page["sin_sq.x"])
    a = x ** 2
    y = a.sin()
    y.backward()
    assert round(a.grad, 3) == page["sin_sq.dy_da"]
    assert round(x.grad, 3) == page["sin_sq.dy_dx"]
    assert x.grad == pytest.approx(math.cos(4.0) * 4.0, rel=1e-15)
    # forward mode with dual numbers reaches the same derivative
    d = dual_derivative(lambda t: (t ** 2).sin(), 2.0)
    assert d == pytest.approx(x.grad, rel=1e-15)


def test_polynomial_relu_and_exercises(page):
    x = Var(2.0)
    y = x ** 2 + 3 * x + 1
    y.backward()
    assert x.grad == page["poly.dy_dx"]

    x1, x2 = Var(2.0), Var(3.0)
    y = (x1 * x2 + Var(1.0)).relu()
    y.backward()
    assert (y.value, x1.grad, x2.grad) == (page["relu1.y"], page["relu1.dy_dx1"], page["relu1.dy_dx2"])

    a, b, c = Var(2.0), Var(-3.0), Var(10.0)
    f = (a * b + c).relu()
    f.backward()
    assert (f.value, a.grad, b.grad, c.grad) == (page["relu2.f"], page["relu2.df_da"],
                                                 page["relu2.df_db"], page["relu2.df_dc"])
    # negative relu input: every gradient is zero (exercise 3's hint)
    w1, w2, bb = Var(-1.0), Var(-1.0), Var(-0.5)
    r = (w1 * 1.0 + w2 * 2.0 + bb).relu()
    r.backward()
    assert (w1.grad, w2.grad, bb.grad) == (0.0, 0.0, 0.0)

    x = Var(2.0)
    (x ** 3).backward()
    assert x.grad == page["cube.dy_dx"]
    for x0, key in ((0.0, "tanh.d0"), (2.0, "tanh.d2")):
        x = Var(x0)
        x.tanh().backward()
        assert round(x.grad, 4) == page[key]


def test_ad_gradient_check(page):
    def expr(v):
        return (v ** 3 + v * 2 + 1).tanh()

    x = Var(page["gradcheck_ad.x"])
    expr(x).backward()
    h = 1e-7
    num = (math.tanh((0.5 + h) ** 3 + 2 * (0.5 + h) + 1) - math.tanh((0.5 - h) ** 3 + 2 * (0.5 - h) + 1)) / (2 * h)
    assert abs(x.grad - num) < page["gradcheck_ad.bound"]
    assert dual_derivative(lambda t: (t ** 3 + t * 2 + 1).tanh(), 0.5) == pytest.approx(x.grad, rel=1e-14)


def _xor_run(seed, steps, lr=0.05):
    """[2, 4, 1] tanh MLP on XOR with sum-of-squares loss and plain SGD ([AD] Step 5)."""
    rng = random.Random(seed)
    layers = []
    for nin, nout in ((2, 4), (4, 1)):
        layers.append([([Var(rng.uniform(-1, 1)) for _ in range(nin)], Var(0.0)) for _ in range(nout)])
    params = [p for layer in layers for (ws, b) in layer for p in ws + [b]]

    def model(x):
        for layer in layers:
            x = [vsum([wi * xi for wi, xi in zip(ws, x)] + [b]).tanh() for ws, b in layer]
        return x[0]

    xs = [[0, 0], [0, 1], [1, 0], [1, 1]]
    ys = [-1, 1, 1, -1]
    losses = []
    for _ in range(steps):
        loss = vsum([(model(x) - y) ** 2 for x, y in zip(xs, ys)])
        for p in params:
            p.grad = 0.0
        loss.backward()
        for p in params:
            p.value -= lr * p.grad
        losses.append(loss.value)
    preds = [model(x).value for x in xs]
    return losses, preds


def test_xor_mlp_learns():
    # The page prints no run; the checks are qualitative: the loss falls over the first
    # 100 steps, and longer training gets all four signs right.
    losses, _ = _xor_run(seed=42, steps=100)
    assert losses[-1] < losses[0]
    losses, preds = _xor_run(seed=42, steps=2000)
    assert all(np.sign(p) == y for p, y in zip(preds, [-1, 1, 1, -1])), preds
    assert losses[-1] < 0.1
