"""Oracle trainers of the pages' two small networks, float64.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the product path.

[LM1] "Build a language model in C# from scratch (1)", "Training loop": a 2 -> 16 -> 2
network (tanh hidden layer, softmax cross-entropy over two classes) learns whether a point
lies inside the circle x^2 + y^2 < 0.5; SGD or AdamW, lr 0.05, no weight decay; the loop runs
steps 0 .. 500 inclusive, each one forward, loss, zeroed gradients, backward, update.
[AD] "Chain rule and automatic differentiation", Step 5: a [2, 4, 1] MLP of tanh neurons learns
XOR (targets -1 / 1) with the sum of squared errors and plain SGD, lr 0.05.

Both are written with the tensor ops of oracle.ops (their forward and backward rules), the
weights stored [in, out] as the pages' Linear layers are.
"""
from __future__ import annotations

import numpy as np

from . import ops


def train_circle(xs, ys, w1, b1, w2, b2, opt: str, lr: float = 0.05, steps: int = 500):
    """Runs steps + 1 iterations (0 .. steps); returns per-iteration (loss, accuracy) measured
    before that iteration's update, and the final parameters."""
    xs = ops._f64(xs)
    ys = np.asarray(ys)
    p = [ops._f64(t).copy() for t in (w1, b1, w2, b2)]
    m = [np.zeros_like(t) for t in p]
    v = [np.zeros_like(t) for t in p]
    losses, accs = [], []
    for step in range(steps + 1):
        w1_, b1_, w2_, b2_ = p
        h = ops.tanh_fwd(ops.add_fwd(ops.matmul_fwd(xs, w1_), b1_))
        logits = ops.add_fwd(ops.matmul_fwd(h, w2_), b2_)
        loss, lse = ops.softmax_ce_fwd(logits, ys)
        losses.append(loss)
        accs.append(float(np.mean(np.argmax(logits, axis=-1) == ys)))
        dlogits = ops.softmax_ce_bwd(logits, ys, lse)
        dh, dw2 = ops.matmul_bwd(h, w2_, dlogits)
        db2 = ops.add_bwd(dlogits, b2_.shape)[1]
        da1 = ops.tanh_bwd(h, dh)
        _, dw1 = ops.matmul_bwd(xs, w1_, da1)
        db1 = ops.add_bwd(da1, b1_.shape)[1]
        grads = [dw1, db1, dw2, db2]
        for i in range(4):
            if opt == "sgd":
                p[i] = ops.sgd(p[i], grads[i], lr)
            else:
                p[i], m[i], v[i] = ops.adamw(p[i], grads[i], m[i], v[i], step + 1, lr, wd=0.0)
    return np.array(losses), np.array(accs), p


def train_xor(xs, ys, w1, b1, w2, b2, lr: float = 0.05, steps: int = 100):
    """Returns the loss of every step (before its update) and the final predictions [4, 1]."""
    xs, ys = ops._f64(xs), ops._f64(ys)
    p = [ops._f64(t).copy() for t in (w1, b1, w2, b2)]

    def forward(w1_, b1_, w2_, b2_):
        h = ops.tanh_fwd(ops.add_fwd(ops.matmul_fwd(xs, w1_), b1_))
        return h, ops.tanh_fwd(ops.add_fwd(ops.matmul_fwd(h, w2_), b2_))

    losses = []
    for _ in range(steps):
        w1_, b1_, w2_, b2_ = p
        h, pred = forward(*p)
        d = ops.add_fwd(pred, ops.scale_fwd(ys, -1.0))
        sq = ops.mul_fwd(d, d)
        losses.append(ops.sum_fwd(sq))
        dsq = ops.sum_bwd(sq.shape, 1.0)
        dd_a, dd_b = ops.mul_bwd(d, d, dsq)  # d appears twice: both contributions add
        dpred = ops.add_bwd(dd_a + dd_b, ())[0]
        da2 = ops.tanh_bwd(pred, dpred)
        dh, dw2 = ops.matmul_bwd(h, w2_, da2)
        db2 = ops.add_bwd(da2, b2_.shape)[1]
        da1 = ops.tanh_bwd(h, dh)
        _, dw1 = ops.matmul_bwd(xs, w1_, da1)
        db1 = ops.add_bwd(da1, b1_.shape)[1]
        p = [ops.sgd(t, g, lr) for t, g in zip(p, (dw1, db1, dw2, db2))]
    return np.array(losses), forward(*p)[1]
