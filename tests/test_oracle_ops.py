"""Pins of the oracle's tensor ops: brute force, library routines, invariants, the scalar
reverse-mode engine and finite differences. None of them re-types an oracle formula."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import ops
from oracle.scalar_ad import Var, vsum



def _rng(seed):
    return synth.Stream(seed)


def _normal(st, *shape, std=1.0):
    return st.normal(int(np.prod(shape)), std).reshape(shape).astype(np.float64)


def _rel(a, b):
    a, b = np.ravel(a), np.ravel(b)
    den = np.linalg.norm(a) + np.linalg.norm(b)
    return 0.0 if den == 0 else np.linalg.norm(a - b) / den


def _fd_check(f, inputs, grads, h=1e-6, proj_seed=5):
    """Central-difference check of analytic grads of sum(f(inputs) * R), fixed random R
    ([LM1] "Gradient Check": a tensor output is reduced with a fixed random projection)."""
    out = f(*inputs)
    R = _normal(_rng(proj_seed), *np.shape(out))
    worst = 0.0
    for x, g in zip(inputs, grads):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = x[i]
            x[i] = old + h
            lp = (f(*inputs) * R).sum()
            x[i] = old - h
            lm = (f(*inputs) * R).sum()
            x[i] = old
            num[i] = (lp - lm) / (2 * h)
        worst = max(worst, _rel(g(R), num))
    return worst


# ----------------------------------------------------------------------- MatMul
def test_matmul_brute_force_and_fd():
    st = _rng(11)
    x, w = _normal(st, 3, 5), _normal(st, 5, 4)
    y = ops.matmul_fwd(x, w)
    for i in range(3):
        for j in range(4):
            assert y[i, j] == pytest.approx(sum(x[i, p] * w[p, j] for p in range(5)), rel=1e-13)
    f = lambda a, b: ops.matmul_fwd(a, b)
    rel = _fd_check(f, [x, w], [lambda R: ops.matmul_bwd(x, w, R)[0], lambda R: ops.matmul_bwd(x, w, R)[1]])
    assert rel < 1e-8
    # MatMulT is MatMul with an explicitly transposed weight
    wt = np.ascontiguousarray(w.T)
    np.testing.assert_allclose(ops.matmul_t_fwd(x, wt), y, rtol=1e-14)
    g = _normal(st, 3, 4)
    dx_t, dw_t = ops.matmul_t_bwd(x, wt, g)
    dx, dw = ops.matmul_bwd(x, w, g)
    np.testing.assert_allclose(dx_t, dx, rtol=1e-13)
    np.testing.assert_allclose(dw_t, dw.T, rtol=1e-13)
    rel = _fd_check(lambda a, b: ops.matmul_t_fwd(a, b), [x, wt],
                    [lambda R: ops.matmul_t_bwd(x, wt, R)[0], lambda R: ops.matmul_t_bwd(x, wt, R)[1]])
    assert rel < 1e-8


def test_matmul_against_scalar_engine():
    st = _rng(12)
    x, w = _normal(st, 2, 3), _normal(st, 3, 2)
    g = _normal(st, 2, 2)
    X = [[Var(v) for v in row] for row in x]
    W = [[Var(v) for v in row] for row in w]
    loss = vsum(vsum(X[i][p] * W[p][j] for p in range(3)) * g[i, j] for i in range(2) for j in range(2))
    loss.backward()
    dx, dw = ops.matmul_bwd(x, w, g)
    np.testing.assert_allclose([[v.grad for v in r] for r in X], dx, rtol=1e-13)
    np.testing.assert_allclose([[v.grad for v in r] for r in W], dw, rtol=1e-13)


def test_bias_grad_is_column_sum():
    g = np.arange(12.0).reshape(4, 3)
    np.testing.assert_array_equal(ops.bias_bwd(g), [18.0, 22.0, 26.0])


# -------------------------------------------------------------------- LayerNorm
def test_layernorm_against_torch_and_invariants():
    st = _rng(13)
    x = _normal(st, 7, 33) * 3 + 1.5
    gamma, beta = _normal(st, 33), _normal(st, 33)
    y, mean, rstd = ops.layernorm_fwd(x, gamma, beta)
    ref = torch.nn.functional.layer_norm(torch.tensor(x), (33,), torch.tensor(gamma), torch.tensor(beta), 1e-5)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    y1, _, _ = ops.layernorm_fwd(x, np.ones(33), np.zeros(33))
    var = x.var(axis=1)
    np.testing.assert_allclose(y1.mean(axis=1), 0, atol=1e-13)
    np.testing.assert_allclose(y1.var(axis=1), var / (var + 1e-5), rtol=1e-12)
    g = _normal(st, 7, 33)
    dx, dg, db = ops.layernorm_bwd(x, gamma, mean, rstd, g)
    xt = torch.tensor(x, requires_grad=True)
    gt, bt = torch.tensor(gamma, requires_grad=True), torch.tensor(beta, requires_grad=True)
    (torch.nn.functional.layer_norm(xt, (33,), gt, bt, 1e-5) * torch.tensor(g)).sum().backward()
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(db, bt.grad.numpy(), rtol=1e-10, atol=1e-12)
    # per-row invariants of the input gradient
    xhat = (x - mean[:, None]) * rstd[:, None]
    np.testing.assert_allclose(dx.sum(axis=1), 0, atol=1e-11)
    # sum(dx * xhat) = rstd * sum(g gamma xhat) * (1 - mean(xhat^2)), which is 0 only at eps = 0
    expect = rstd * (g * gamma * xhat).sum(axis=1) * (1 - (xhat ** 2).mean(axis=1))
    np.testing.assert_allclose((dx * xhat).sum(axis=1), expect, rtol=1e-6, atol=1e-13)


def test_layernorm_against_scalar_engine_and_fd():
    st = _rng(14)
    x = _normal(st, 2, 5)
    gamma, beta = _normal(st, 5), _normal(st, 5)
    g = _normal(st, 2, 5)
    X = [[Var(v) for v in r] for r in x]
    G = [Var(v) for v in gamma]
    Bb = [Var(v) for v in beta]
    terms = []
    for i in range(2):
        mu = vsum(X[i]) / 5
        var = vsum((xv - mu) ** 2 for xv in X[i]) / 5
        r = 1 / (var + 1e-5).sqrt()
        terms += [((X[i][c] - mu) * r * G[c] + Bb[c]) * g[i, c] for c in range(5)]
    vsum(terms).backward()
    _, mean, rstd = ops.layernorm_fwd(x, gamma, beta)
    dx, dg, db = ops.layernorm_bwd(x, gamma, mean, rstd, g)
    np.testing.assert_allclose([[v.grad for v in r] for r in X], dx, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose([v.grad for v in G], dg, rtol=1e-12)
    np.testing.assert_allclose([v.grad for v in Bb], db, rtol=1e-12)
    f = lambda a, gm, bt: ops.layernorm_fwd(a, gm, bt)[0]
    bw = lambda R: ops.layernorm_bwd(x, gamma, mean, rstd, R)
    assert _fd_check(f, [x, gamma, beta], [lambda R: bw(R)[0], lambda R: bw(R)[1], lambda R: bw(R)[2]]) < 1e-7


# ------------------------------------------------------------------------- GELU
def test_gelu_special_values_and_library():
    assert ops.gelu_fwd(0.0) == 0.0
    assert ops.gelu_bwd(0.0, 1.0) == 0.5
    x = np.linspace(-6, 6, 241)
    np.testing.assert_allclose(ops.gelu_fwd(x) - ops.gelu_fwd(-x), x, atol=1e-14)
    ref = torch.nn.functional.gelu(torch.tensor(x), approximate="tanh").numpy()
    np.testing.assert_allclose(ops.gelu_fwd(x), ref, rtol=1e-14, atol=1e-15)
    # the tanh form is close to, but not, the erf form
    erf = torch.nn.functional.gelu(torch.tensor(x)).numpy()
    diff = np.abs(ops.gelu_fwd(x) - erf).max()
    assert 1e-5 < diff < 1e-3
    xt = torch.tensor(x, requires_grad=True)
    torch.nn.functional.gelu(xt, approximate="tanh").sum().backward()
    np.testing.assert_allclose(ops.gelu_bwd(x, np.ones_like(x)), xt.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_gelu_against_scalar_engine():
    for x0 in (-2.3, -0.4, 0.0, 0.7, 3.1):
        x = Var(x0)
        u = (x + 0.044715 * x ** 3) * math.sqrt(2 / math.pi)
        (0.5 * x * (1 + u.tanh())).backward()
        assert ops.gelu_bwd(x0, 1.0) == pytest.approx(x.grad, rel=1e-13, abs=1e-15)


# -------------------------------------------------------------------- Embedding
def test_embedding_forward_brute_force():
    st = _rng(15)
    wte, wpe = _normal(st, 9, 4).astype(np.float32), _normal(st, 5, 4).astype(np.float32)
    ids = np.array([[3, 3, 0, 8, 1], [2, 3, 7, 7, 7]])
    x = ops.embedding_fwd(ids, wte, wpe)
    for b in range(2):
        for t in range(5):
            np.testing.assert_array_equal(x[b, t], wte[ids[b, t]].astype(np.float64) + wpe[t])
    with pytest.raises(IndexError):
        ops.embedding_fwd(np.array([[9]]), wte, wpe)


def test_embedding_backward_order_and_fd():
    st = _rng(16)
    B, T, C, V = 3, 4, 6, 5
    ids = np.array([[1, 1, 4, 0], [1, 2, 2, 1], [0, 4, 4, 1]])
    dx = _normal(st, B, T, C).astype(np.float32)
    dwte = _normal(st, V, C).astype(np.float32)
    dwpe = _normal(st, T, C).astype(np.float32)
    exp_te, exp_pe = dwte.copy(), dwpe.copy()
    ops.embedding_bwd(ids, dx, dwte, dwpe)
    # brute force: for each token, float32 adds of its rows in ascending row order
    for v in range(V):
        acc = exp_te[v].copy()
        for r in range(B * T):
            if ids.reshape(-1)[r] == v:
                acc = (acc + dx.reshape(-1, C)[r]).astype(np.float32)
        np.testing.assert_array_equal(dwte[v], acc)
    for t in range(T):
        acc = exp_pe[t].copy()
        for b in range(B):
            acc = (acc + dx[b, t]).astype(np.float32)
        np.testing.assert_array_equal(dwpe[t], acc)
    # derivative check of the scatter in float64 against the forward
    wte, wpe = _normal(st, V, C), _normal(st, T, C)
    R = _normal(st, B, T, C)
    g_te, g_pe = np.zeros((V, C), np.float32), np.zeros((T, C), np.float32)
    ops.embedding_bwd(ids, R, g_te, g_pe)
    h = 1e-6
    for tbl, g in ((wte, g_te), (wpe, g_pe)):
        num = np.zeros_like(tbl)
        for i in np.ndindex(tbl.shape):
            old = tbl[i]
            tbl[i] = old + h
            lp = (ops.embedding_fwd(ids, wte, wpe) * R).sum()
            tbl[i] = old - h
            lm = (ops.embedding_fwd(ids, wte, wpe) * R).sum()
            tbl[i] = old
            num[i] = (lp - lm) / (2 * h)
        assert _rel(g, num) < 1e-6


# -------------------------------------------------------------------- Attention
def test_attention_against_torch_sdpa():
    st = _rng(17)
    B, T, H, hs = 2, 7, 3, 4
    qkv = _normal(st, B, T, 3 * H * hs)
    y, p, lse = ops.attention_fwd(qkv, H)
    q, k, v = (torch.tensor(qkv[..., i * H * hs:(i + 1) * H * hs]).reshape(B, T, H, hs).transpose(1, 2) for i in range(3))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    np.testing.assert_allclose(y, ref.transpose(1, 2).reshape(B, T, H * hs).numpy(), rtol=1e-12, atol=1e-13)
    assert np.all(p[..., np.triu_indices(T, 1)[0], np.triu_indices(T, 1)[1]] == 0.0)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=1e-14)
    dy = _normal(st, B, T, H * hs)
    dqkv = ops.attention_bwd(qkv, p, dy, H)
    qt = torch.tensor(qkv, requires_grad=True)
    qq, kk, vv = (qt[..., i * H * hs:(i + 1) * H * hs].reshape(B, T, H, hs).transpose(1, 2) for i in range(3))
    out = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv, is_causal=True)
    (out.transpose(1, 2).reshape(B, T, H * hs) * torch.tensor(dy)).sum().backward()
    np.testing.assert_allclose(dqkv, qt.grad.numpy(), rtol=1e-10, atol=1e-12)
    # lse is the log of the softmax denominator of the scaled, masked scores
    s = np.einsum("bhid,bhjd->bhij", q.numpy(), k.numpy()) / 2.0
    s[..., np.triu_indices(T, 1)[0], np.triu_indices(T, 1)[1]] = -np.inf
    np.testing.assert_allclose(lse, np.log(np.exp(s).sum(-1)), rtol=1e-13)


def test_attention_special_cases_and_fd():
    st = _rng(18)
    B, T, H, hs = 1, 5, 2, 3
    qkv = _normal(st, B, T, 3 * H * hs)
    y, p, _ = ops.attention_fwd(qkv, H)
    # position 0 sees only itself: its output is its own value row
    np.testing.assert_allclose(y[:, 0], qkv[:, 0, 2 * H * hs:], rtol=1e-14)
    # causality: changing the last token leaves earlier outputs unchanged
    q2 = qkv.copy()
    q2[:, -1] += 1.0
    y2, _, _ = ops.attention_fwd(q2, H)
    np.testing.assert_array_equal(y2[:, :-1], y[:, :-1])
    f = lambda a: ops.attention_fwd(a, H)[0]
    assert _fd_check(f, [qkv], [lambda R: ops.attention_bwd(qkv, p, R, H)]) < 1e-7


# -------------------------------------------------------- Softmax cross-entropy
def test_softmax_ce_closed_forms_and_library():
    n, V = 6, 11
    loss, lse = ops.softmax_ce_fwd(np.zeros((n, V)), np.arange(n) % V)
    assert loss == pytest.approx(math.log(V), rel=1e-15)
    # V = 2 is the logistic loss log(1 + exp(-margin))
    z = np.array([[0.3, -1.2], [2.0, 0.5], [-0.7, 0.1]])
    t = np.array([0, 1, 1])
    margin = np.where(t == 0, z[:, 0] - z[:, 1], z[:, 1] - z[:, 0])
    assert ops.softmax_ce_fwd(z, t)[0] == pytest.approx(np.mean(np.log1p(np.exp(-margin))), rel=1e-14)
    st = _rng(19)
    x = _normal(st, 9, 13) * 4
    tg = np.array([0, 12, 5, 5, 3, 7, 1, 11, 2])
    loss, lse = ops.softmax_ce_fwd(x, tg)
    xt = torch.tensor(x, requires_grad=True)
    ref = torch.nn.functional.cross_entropy(xt, torch.tensor(tg))
    assert loss == pytest.approx(ref.item(), rel=1e-14)
    (ref * 0.75).backward()
    d = ops.softmax_ce_bwd(x, tg, lse, 0.75)
    np.testing.assert_allclose(d, xt.grad.numpy(), rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(d.sum(axis=1), 0, atol=1e-15)


def test_softmax_ce_against_scalar_engine():
    x = np.array([[0.2, -0.5, 1.1], [2.0, 0.0, -1.0]])
    t = [2, 0]
    X = [[Var(v) for v in r] for r in x]
    loss = vsum((vsum(v.exp() for v in X[i])).log() - X[i][t[i]] for i in range(2)) / 2
    loss.backward()
    _, lse = ops.softmax_ce_fwd(x, t)
    np.testing.assert_allclose(ops.softmax_ce_bwd(x, t, lse), [[v.grad for v in r] for r in X], rtol=1e-13)


def test_softmax_helper_temperature():
    x = np.array([[1.0, 2.0, 3.0]])
    p = ops.softmax(x, 0.5)
    e = np.exp(np.array([2.0, 4.0, 6.0]))
    np.testing.assert_allclose(p[0], e / e.sum(), rtol=1e-15)


# ------------------------------------------------------------------------ AdamW
def test_adamw_closed_form_constant_gradient():
    # With a constant gradient, mhat = g and vhat = g^2 at every step, so
    # p_t = (1 - a)^t p0 - s (1 - (1 - a)^t) / a with a = lr wd and s = lr g / (|g| + eps).
    lr, wd, eps, g, p0 = 1e-2, 0.1, 1e-8, -0.37, 0.8
    p, m, v = p0, 0.0, 0.0
    for t in range(1, 51):
        p, m, v = ops.adamw(p, g, m, v, t, lr, 0.9, 0.999, eps, wd)
        a, s = lr * wd, lr * g / (abs(g) + eps)
        assert float(p) == pytest.approx((1 - a) ** t * p0 - s * (1 - (1 - a) ** t) / a, rel=1e-12)
    p, m, v = p0, 0.0, 0.0
    for t in range(1, 21):
        p, m, v = ops.adamw(p, g, m, v, t, lr, 0.9, 0.999, eps, 0.0)
    assert float(p) == pytest.approx(p0 - 20 * lr * g / (abs(g) + eps), rel=1e-12)


def test_adamw_against_torch():
    st = _rng(20)
    p0 = _normal(st, 40)
    grads = [_normal(st, 40) for _ in range(5)]
    pt = torch.tensor(p0, requires_grad=True)
    opt = torch.optim.AdamW([pt], lr=3e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.05)
    p, m, v = p0.copy(), np.zeros(40), np.zeros(40)
    for t, g in enumerate(grads, 1):
        pt.grad = torch.tensor(g)
        opt.step()
        p, m, v = ops.adamw(p, g, m, v, t, 3e-3, 0.9, 0.999, 1e-8, 0.05)
    np.testing.assert_allclose(p, pt.detach().numpy(), rtol=1e-13, atol=1e-15)


def test_fp32_gradcheck_setting_of_the_page(page):
    """The page's own setting (float32, h = 1e-2, relative error < 1e-3) on each op."""
    st = _rng(21)
    h, thr = page["gradcheck.h"], page["gradcheck.threshold"]

    def fd32(f, x, analytic):
        x = x.astype(np.float32)
        R = _normal(_rng(22), *np.shape(f(x))).astype(np.float32)
        num = np.zeros(x.shape)
        for i in np.ndindex(x.shape):
            old = x[i]
            x[i] = old + np.float32(h)
            lp = np.float32((f(x).astype(np.float32) * R).sum(dtype=np.float32))
            x[i] = old - np.float32(h)
            lm = np.float32((f(x).astype(np.float32) * R).sum(dtype=np.float32))
            x[i] = old
            num[i] = (lp - lm) / (2 * h)
        return _rel(analytic(x, R), num)

    x = _normal(st, 4, 6)
    w = _normal(st, 6, 3)
    gm, bt = _normal(st, 6), _normal(st, 6)
    assert fd32(lambda a: ops.matmul_fwd(a, w), x, lambda a, R: ops.matmul_bwd(a, w, R)[0]) < thr
    assert fd32(ops.gelu_fwd, x, lambda a, R: ops.gelu_bwd(a, R)) < thr

    def ln_an(a, R):
        _, mu, rs = ops.layernorm_fwd(a, gm, bt)
        return ops.layernorm_bwd(a, gm, mu, rs, R)[0]

    assert fd32(lambda a: ops.layernorm_fwd(a, gm, bt)[0], x, ln_an) < thr
    qkv = _normal(st, 1, 4, 6)
    assert fd32(lambda a: ops.attention_fwd(a, 2)[0], qkv,
                lambda a, R: ops.attention_bwd(a, ops.attention_fwd(a, 2)[1], R, 2)) < thr
    tg = np.array([1, 0, 5, 2])
    assert fd32(lambda a: np.array(ops.softmax_ce_fwd(a, tg)[0]), x,
                lambda a, R: ops.softmax_ce_bwd(a, tg, ops.softmax_ce_fwd(a, tg)[1], float(R))) < thr
