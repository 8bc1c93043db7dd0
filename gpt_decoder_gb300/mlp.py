"""The pages' two small networks trained on the GPU through libgk's generic ops.

[LM1] "Build a language model in C# from scratch (1)", "Training loop": a 2 -> 16 -> 2 network,
logits = Add(MatMul(Tanh(Add(MatMul(xs, w1), b1)), w2), b2), softmax cross-entropy over two
classes (is the point inside x^2 + y^2 < 0.5), SGD or AdamW at lr 0.05 without decay, steps
0 .. 500 each doing forward, loss, zeroed gradients, backward, update.
[AD] "Chain rule and automatic differentiation", Step 5: a [2, 4, 1] MLP of tanh neurons on XOR
(targets -1 / 1), loss Sum(Mul(d, d)) with d = Add(pred, Scale(y, -1)), plain SGD at lr 0.05.

Every forward and backward op runs in libgk kernels (gk_matmul_*, gk_add_*, gk_tanh_*,
gk_mul_*, gk_scale_*, gk_sum_*, gk_softmax_ce_*, gk_sgd_step, gk_adamw_step); this module
holds the device buffers and the order of the calls (gradient zeroing and the logits history
are memory operations on the current torch stream, which `ctx` must be bound to). Weights are
stored [in, out].
"""
from __future__ import annotations

import numpy as np

from . import gk


def _dev(a, dtype=None):
    import torch

    t = torch.as_tensor(np.ascontiguousarray(a))
    return t.to(device="cuda", dtype=dtype or t.dtype).contiguous()


class _Params:
    """Parameters, gradients and AdamW moments of a list of float32 tensors."""

    def __init__(self, tensors):
        import torch

        self.p = [_dev(np.asarray(t, np.float32)) for t in tensors]
        self.g = [torch.zeros_like(t) for t in self.p]
        self.m = [torch.zeros_like(t) for t in self.p]
        self.v = [torch.zeros_like(t) for t in self.p]

    def zero_grad(self):
        for g in self.g:
            g.zero_()

    def step(self, ctx, opt, lr, t):
        if opt == "sgd":
            for p, g in zip(self.p, self.g):
                gk.gk_sgd_step(ctx, p, g, p.numel(), lr)
        else:
            blocks = [dict(p=p, g=g, m=m, v=v, n=p.numel(), decay=0) for p, g, m, v in zip(self.p, self.g, self.m, self.v)]
            gk.gk_adamw_step(ctx, blocks, lr, 0.9, 0.999, 1e-8, 0.0, t)

    def host(self):
        return [p.cpu().numpy() for p in self.p]


def train_circle(ctx, xs, ys, w1, b1, w2, b2, opt="sgd", lr=0.05, steps=500):
    """Returns (loss [steps + 1], accuracy [steps + 1], final parameters): iteration i's loss
    and accuracy are taken before its update."""
    import torch

    n, H = xs.shape[0], w1.shape[1]
    x, y = _dev(np.asarray(xs, np.float32)), _dev(np.asarray(ys, np.int32))
    P = _Params([w1, b1, w2, b2])
    w1_, b1_, w2_, b2_ = P.p
    gw1, gb1, gw2, gb2 = P.g
    f = lambda *s: torch.empty(*s, device="cuda")
    a1, h, logits, dlogits, dh = f(n, H), f(n, H), f(n, 2), f(n, 2), f(n, H)
    lse, losses, hist = f(n), f(steps + 1), f(steps + 1, n, 2)
    F32 = gk.GK_F32
    for step in range(steps + 1):
        # forward: h = tanh(xs w1 + b1), logits = h w2 + b2, loss = CE(logits, ys)
        gk.gk_matmul_fwd(ctx, F32, x, 2, w1_, H, 0, None, None, 0, a1, H, F32, n, 2, H)
        gk.gk_add_fwd(ctx, a1, b1_, a1, n * H, H)
        gk.gk_tanh_fwd(ctx, a1, h, n * H)
        gk.gk_matmul_fwd(ctx, F32, h, H, w2_, 2, 0, None, None, 0, logits, 2, F32, n, H, 2)
        gk.gk_add_fwd(ctx, logits, b2_, logits, n * 2, 2)
        gk.gk_softmax_ce_fwd(ctx, logits, 2, y, losses[step:], lse, n, 2)
        hist[step].copy_(logits)
        # zeroed gradients, backward
        P.zero_grad()
        gk.gk_softmax_ce_bwd(ctx, logits, 2, y, lse, None, dlogits, 2, F32, n, 2)
        gk.gk_add_bwd(ctx, dlogits, None, gb2, n * 2, 2, 1)
        gk.gk_matmul_bwd(ctx, F32, h, H, w2_, 2, 0, dlogits, 2, dh, H, F32, 0, None, 0, gw2, 2, None, n, H, 2)
        gk.gk_tanh_bwd(ctx, h, dh, dh, n * H, 0)
        gk.gk_add_bwd(ctx, dh, None, gb1, n * H, H, 1)
        gk.gk_matmul_bwd(ctx, F32, x, 2, w1_, H, 0, dh, H, None, 0, F32, 0, None, 0, gw1, H, None, n, 2, H)
        P.step(ctx, opt, lr, step + 1)
    gk.gk_sync(ctx)
    lg = hist.cpu().numpy()
    acc = (lg.argmax(axis=-1) == np.asarray(ys)[None, :]).mean(axis=-1)
    return losses.cpu().numpy(), acc, P.host()


def train_xor(ctx, xs, ys, w1, b1, w2, b2, lr=0.05, steps=100):
    """Returns (loss of every step before its update, final predictions [4, 1])."""
    import torch

    H = w1.shape[1]
    x, yt = _dev(np.asarray(xs, np.float32)), _dev(np.asarray(ys, np.float32))
    P = _Params([w1, b1, w2, b2])
    w1_, b1_, w2_, b2_ = P.p
    gw1, gb1, gw2, gb2 = P.g
    f = lambda *s: torch.empty(*s, device="cuda")
    a1, h, pred, negy, d, sq, dsq, dd, dpred, dh = (f(4, H), f(4, H), f(4, 1), f(4, 1), f(4, 1), f(4, 1), f(4, 1),
                                                    f(4, 1), f(4, 1), f(4, H))
    one, losses = torch.ones(1, device="cuda"), f(steps)
    F32 = gk.GK_F32

    def forward():
        gk.gk_matmul_fwd(ctx, F32, x, 2, w1_, H, 0, None, None, 0, a1, H, F32, 4, 2, H)
        gk.gk_add_fwd(ctx, a1, b1_, a1, 4 * H, H)
        gk.gk_tanh_fwd(ctx, a1, h, 4 * H)
        gk.gk_matmul_fwd(ctx, F32, h, H, w2_, 1, 0, None, None, 0, pred, 1, F32, 4, H, 1)
        gk.gk_add_fwd(ctx, pred, b2_, pred, 4, 1)
        gk.gk_tanh_fwd(ctx, pred, pred, 4)

    gk.gk_scale_fwd(ctx, yt, -1.0, negy, 4)
    for step in range(steps):
        forward()
        gk.gk_add_fwd(ctx, pred, negy, d, 4, 4)          # d = pred - y
        gk.gk_mul_fwd(ctx, d, d, sq, 4)                  # d^2
        gk.gk_sum_fwd(ctx, sq, losses[step:], 4)         # loss
        P.zero_grad()
        gk.gk_sum_bwd(ctx, one, dsq, 4, 0)
        gk.gk_mul_bwd(ctx, dsq, d, d, dd, None, 4, 0)   # d is both factors: both rules add
        gk.gk_mul_bwd(ctx, dsq, d, d, None, dd, 4, 1)
        gk.gk_add_bwd(ctx, dd, dpred, None, 4, 4, 0)
        gk.gk_tanh_bwd(ctx, pred, dpred, dpred, 4, 0)
        gk.gk_add_bwd(ctx, dpred, None, gb2, 4, 1, 1)
        gk.gk_matmul_bwd(ctx, F32, h, H, w2_, 1, 0, dpred, 1, dh, H, F32, 0, None, 0, gw2, 1, None, 4, H, 1)
        gk.gk_tanh_bwd(ctx, h, dh, dh, 4 * H, 0)
        gk.gk_add_bwd(ctx, dh, None, gb1, 4 * H, H, 1)
        gk.gk_matmul_bwd(ctx, F32, x, 2, w1_, H, 0, dh, H, None, 0, F32, 0, None, 0, gw1, H, None, 4, 2, H)
        P.step(ctx, "sgd", lr, step + 1)
    forward()
    gk.gk_sync(ctx)
    return losses.cpu().numpy(), pred.cpu().numpy()
