"""A scalar reverse-mode automatic differentiator: the oracle's independent derivative check.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the product path.

[AD] "Forward mode vs reverse mode" and "Building an Autograd engine": every operation
records its inputs and its local derivatives; backward seeds d(out)/d(out) = 1 and walks
the recorded graph in reverse topological order, ADDING each contribution into the
inputs' gradients ([LM1] "Why += and not =").

Design (not the pages' closure-based one): each node keeps (parent, local derivative)
pairs and a creation serial number. A parent is always created before its child, so
decreasing serial number is a reverse topological order; backward sorts the reachable
nodes by it. Pure Python floats, so only tiny graphs are practical.

The tensor ops' hand-derived backward rules in ``oracle.ops`` are checked against this
engine on tiny inputs: the two share no formula, only the forward definition.
"""
from __future__ import annotations

import itertools
import math

_serial = itertools.count()


class Var:
    __slots__ = ("value", "grad", "parents", "serial")

    def __init__(self, value, parents=()):
        self.value = float(value)
        self.grad = 0.0
        self.parents = tuple(parents)  # ((Var, d self / d parent), ...)
        self.serial = next(_serial)

    # -- arithmetic -------------------------------------------------------------
    def __add__(self, o):
        o = lift(o)
        return Var(self.value + o.value, ((self, 1.0), (o, 1.0)))

    __radd__ = __add__

    def __neg__(self):
        return Var(-self.value, ((self, -1.0),))

    def __sub__(self, o):
        o = lift(o)
        return Var(self.value - o.value, ((self, 1.0), (o, -1.0)))

    def __rsub__(self, o):
        return lift(o) - self

    def __mul__(self, o):
        o = lift(o)
        return Var(self.value * o.value, ((self, o.value), (o, self.value)))

    __rmul__ = __mul__

    def __truediv__(self, o):
        o = lift(o)
        return Var(self.value / o.value,
                   ((self, 1.0 / o.value), (o, -self.value / (o.value * o.value))))

    def __rtruediv__(self, o):
        return lift(o) / self

    def __pow__(self, n):
        assert not isinstance(n, Var), "only constant exponents"
        return Var(self.value ** n, ((self, n * self.value ** (n - 1)),))

    # -- elementary functions ---------------------------------------------------
    def exp(self):
        e = math.exp(self.value)
        return Var(e, ((self, e),))

    def log(self):
        return Var(math.log(self.value), ((self, 1.0 / self.value),))

    def tanh(self):
        t = math.tanh(self.value)
        return Var(t, ((self, 1.0 - t * t),))

    def sin(self):
        return Var(math.sin(self.value), ((self, math.cos(self.value)),))

    def cos(self):
        return Var(math.cos(self.value), ((self, -math.sin(self.value)),))

    def sqrt(self):
        r = math.sqrt(self.value)
        return Var(r, ((self, 0.5 / r),))

    def relu(self):
        return Var(max(0.0, self.value), ((self, 1.0 if self.value > 0 else 0.0),))

    # -- reverse sweep -------------------------------------------------------------
    def backward(self):
        """Seed this node's gradient with 1 and propagate to every reachable input."""
        seen, stack, nodes = set(), [self], []
        while stack:
            n = stack.pop()
            if id(n) in seen:
                continue
            seen.add(id(n))
            nodes.append(n)
            stack.extend(p for p, _ in n.parents)
        nodes.sort(key=lambda n: n.serial, reverse=True)
        self.grad += 1.0
        for n in nodes:
            for p, d in n.parents:
                p.grad += d * n.grad


def lift(x):
    return x if isinstance(x, Var) else Var(x)


def vsum(xs):
    out = Var(0.0)
    for x in xs:
        out = out + x
    return out


def dual_derivative(f, x0):
    """Forward-mode derivative of f at x0 with dual numbers (a, a'), a cross-check of
    reverse mode ([AD] "Dual numbers for forward mode"). f takes and returns Dual."""
    return f(Dual(x0, 1.0)).d


class Dual:
    """(value, derivative) pairs with the product rule (a, a')(b, b') = (ab, a'b + ab')."""

    __slots__ = ("v", "d")

    def __init__(self, v, d=0.0):
        self.v, self.d = float(v), float(d)

    def __add__(self, o):
        o = o if isinstance(o, Dual) else Dual(o)
        return Dual(self.v + o.v, self.d + o.d)

    __radd__ = __add__

    def __mul__(self, o):
        o = o if isinstance(o, Dual) else Dual(o)
        return Dual(self.v * o.v, self.d * o.v + self.v * o.d)

    __rmul__ = __mul__

    def __pow__(self, n):
        return Dual(self.v ** n, n * self.v ** (n - 1) * self.d)

    def sin(self):
        return Dual(math.sin(self.v), math.cos(self.v) * self.d)

    def tanh(self):
        t = math.tanh(self.v)
        return Dual(t, (1 - t * t) * self.d)
