"""Oracle definitions of the tensor ops of the decoder step, forward and backward.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the product path.

Conventions (from [LM1] "The Tensor class"): every tensor is a row-major array; a Linear
weight is stored [in, out]; backward rules ADD into gradient buffers ([LM1] "Why += and
not ="), so the functions here return the contribution and the caller adds it.
Arithmetic is float64 throughout unless a function says otherwise.
"""
from __future__ import annotations

import math

import numpy as np

F64 = np.float64

# Tanh-approximate GELU constants: sqrt(2/pi) and the cubic coefficient of the published
# approximation (Hendrycks & Gimpel, "Gaussian Error Linear Units", 2016). The pages name
# the tanh form ("gelu_new") but do not print its constants.
GELU_K = math.sqrt(2.0 / math.pi)
GELU_C = 0.044715

LN_EPS = 1e-5


def _f64(a):
    return np.asarray(a, dtype=F64)


# --------------------------------------------------------------------------- MatMul
def matmul_fwd(x, w):
    """Y = X W for X [n, k] and W [k, m].

    [LM1] "Ops: forward computation and backward rule for each op", MatMul listing.
    """
    return _f64(x) @ _f64(w)


def matmul_bwd(x, w, g):
    """Contributions dX = G W^T and dW = X^T G of Y = X W.

    [LM1] "Ops: forward computation and backward rule for each op", MatMul backward rule
    (the shape argument there fixes which side each transpose goes on).
    """
    g = _f64(g)
    return g @ _f64(w).T, _f64(x).T @ g


def matmul_t_fwd(x, w):
    """Y = X W^T for X [n, k] and W [m, k] (MatMulT, the tied LM head).

    [LM1] "Ops..." op table (MatMulT, used for GPT-2's last layer); [LM4] "Loading weights
    into our classes" (weight tying: the logits use the token table wte).
    """
    return _f64(x) @ _f64(w).T


def matmul_t_bwd(x, w, g):
    """Contributions dX = G W and dW = G^T X of Y = X W^T."""
    g = _f64(g)
    return g @ _f64(w), g.T @ _f64(x)


def bias_bwd(g):
    """Gradient of a bias broadcast over rows: the column sum of G.

    [LM1] "Ops..." op table (Add with broadcast) and "Gradient Check" (Add broadcast bias).
    """
    return _f64(g).sum(axis=0)


# ------------------------------------------------------------------------ LayerNorm
def layernorm_fwd(x, gamma, beta, eps=LN_EPS):
    """y = (x - mean) * rstd * gamma + beta per row, rstd = 1 / sqrt(var + eps).

    [LM1] "Ops..." op table (LayerNorm); [LM4] "A first prediction" / loading (ln_1, ln_2,
    ln_f carry a weight and a bias). Reading: the pages print no formula; the variance is
    the biased (population) one, the GPT-2 convention, and eps is 1e-5.
    Returns (y, mean, rstd) with mean and rstd per row.
    """
    x = _f64(x)
    mean = x.mean(axis=-1)
    var = ((x - mean[..., None]) ** 2).mean(axis=-1)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mean[..., None]) * rstd[..., None]
    return xhat * _f64(gamma) + _f64(beta), mean, rstd


def layernorm_bwd(x, gamma, mean, rstd, g):
    """(dx, dgamma, dbeta) of layernorm_fwd for upstream gradient g.

    With xhat = (x - mean) rstd and gh = g * gamma, each row gives
    dx = rstd (gh - mean(gh) - xhat mean(gh xhat)); dgamma = sum_rows g xhat; dbeta = sum_rows g.
    This is the chain rule through mean, variance and scale (no approximation).
    """
    x, g = _f64(x), _f64(g)
    mean, rstd = _f64(mean), _f64(rstd)
    xhat = (x - mean[..., None]) * rstd[..., None]
    gh = g * _f64(gamma)
    dx = rstd[..., None] * (gh - gh.mean(axis=-1, keepdims=True)
                            - xhat * (gh * xhat).mean(axis=-1, keepdims=True))
    red = tuple(range(x.ndim - 1))
    return dx, (g * xhat).sum(axis=red), g.sum(axis=red)


# ----------------------------------------------------------------------------- GELU
def gelu_fwd(x):
    """GELU in its tanh form: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).

    [LM4] "Common mistakes" and the HF comparison: GPT-2 uses the tanh approximation
    ("gelu_new"); the exact erf form is named as the mistake.
    """
    x = _f64(x)
    return 0.5 * x * (1.0 + np.tanh(GELU_K * (x + GELU_C * x ** 3)))


def gelu_bwd(x, g):
    """Upstream g times the derivative of gelu_fwd at x (product and chain rules)."""
    x = _f64(x)
    t = np.tanh(GELU_K * (x + GELU_C * x ** 3))
    du = GELU_K * (1.0 + 3.0 * GELU_C * x ** 2)
    return _f64(g) * (0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * du)


# ------------------------------------------------------------------------ Embedding
def embedding_fwd(ids, wte, wpe):
    """x[b, t] = wte[ids[b, t]] + wpe[t] for ids [B, T].

    [LM1] "Ops..." op table (Embedding); [LM4] "Generation with a KV cache" (Gpt.Step adds
    the token row and the position row).
    """
    ids = np.asarray(ids)
    if ids.min(initial=0) < 0 or ids.max(initial=0) >= wte.shape[0]:
        raise IndexError("token id outside the vocabulary")
    T = ids.shape[-1]
    return _f64(wte)[ids] + _f64(wpe)[:T]


def embedding_bwd(ids, dx, dwte, dwpe):
    """Scatter-add dx rows into dwte[ids[r]] and dwpe[r % T], in place, float32.

    [LM1] "Ops..." op table (Embedding) and "Why += and not =": rows that share a token
    accumulate. Reading: an exact comparison needs a defined summation order, so rows are
    taken in ascending flat index r = b*T + t and each add is one float32 addition onto
    the existing gradient value. dwte and dwpe must be float32 arrays; they are modified.
    """
    ids = np.asarray(ids)
    B, T = ids.shape
    dx = np.asarray(dx, dtype=np.float32).reshape(B * T, -1)
    flat = ids.reshape(-1)
    assert dwte.dtype == np.float32 and dwpe.dtype == np.float32
    for r in range(B * T):
        dwte[flat[r]] += dx[r]
        dwpe[r % T] += dx[r]
    return dwte, dwpe


# ------------------------------------------------------------------------ Attention
def split_heads(a, H):
    """[B, T, C] -> [B, H, T, C/H]: head h takes columns [h*hs, (h+1)*hs)."""
    B, T, C = a.shape
    return a.reshape(B, T, H, C // H).transpose(0, 2, 1, 3)


def merge_heads(a):
    """[B, H, T, hs] -> [B, T, H*hs]."""
    B, H, T, hs = a.shape
    return a.transpose(0, 2, 1, 3).reshape(B, T, H * hs)


def attention_fwd(qkv, H):
    """Causal multi-head self-attention from the fused projection qkv [B, T, 3C].

    [LM1] op table (BatchMatMulT, CausalSoftmax, BatchMatMul, Narrow, SplitHeads,
    MergeHeads); [LM4] "Loading weights" (c_attn holds q, k, v side by side, 3C columns)
    and "Generation with a KV cache" (scale 1/sqrt(head size)); [LM4] "The 12 tensors we do
    not use" (row r sees columns 0..r % t: visible = r % t + 1).
    q, k, v are columns [0, C), [C, 2C), [2C, 3C); S = q k^T / sqrt(hs); entries j > i get
    probability exactly 0; P = row softmax(S); y = merge_heads(P v). Reading: no dropout.
    Returns (y [B,T,C], P [B,H,T,T], lse [B,H,T]).
    """
    qkv = _f64(qkv)
    B, T, C3 = qkv.shape
    C = C3 // 3
    hs = C // H
    q, k, v = (split_heads(qkv[..., i * C:(i + 1) * C], H) for i in range(3))
    s = (q @ k.transpose(0, 1, 3, 2)) / math.sqrt(hs)
    mask = np.triu(np.ones((T, T), dtype=bool), k=1)
    s = np.where(mask, -np.inf, s)
    mx = s.max(axis=-1, keepdims=True)
    e = np.exp(s - mx)
    den = e.sum(axis=-1, keepdims=True)
    p = e / den
    lse = (mx + np.log(den))[..., 0]
    return merge_heads(p @ v), p, lse


def attention_bwd(qkv, p, dy, H):
    """dqkv [B, T, 3C] of attention_fwd for upstream dy [B, T, C] and the saved P.

    Chain rule through y = P v, the row softmax and S = q k^T / sqrt(hs):
    dP = dY v^T; dS = P (dP - rowsum(dP P)); dq = dS k / sqrt(hs); dk = dS^T q / sqrt(hs);
    dv = P^T dY. Masked entries have P = 0 and so get no gradient.
    """
    qkv = _f64(qkv)
    B, T, C3 = qkv.shape
    C = C3 // 3
    hs = C // H
    q, k, v = (split_heads(qkv[..., i * C:(i + 1) * C], H) for i in range(3))
    dyh = split_heads(_f64(dy), H)
    dp = dyh @ v.transpose(0, 1, 3, 2)
    ds = p * (dp - (dp * p).sum(axis=-1, keepdims=True))
    scale = 1.0 / math.sqrt(hs)
    dq = (ds @ k) * scale
    dk = (ds.transpose(0, 1, 3, 2) @ q) * scale
    dv = p.transpose(0, 1, 3, 2) @ dyh
    return np.concatenate([merge_heads(dq), merge_heads(dk), merge_heads(dv)], axis=-1)


# ------------------------------------------------------------- Softmax cross-entropy
def softmax_ce_fwd(logits, targets):
    """Mean over rows of (logsumexp(row) - row[target]); also returns the per-row LSE.

    [LM1] "Ops..." SoftmaxCrossEntropy listing: softmax of every row, minus the log of the
    target's probability, averaged over all rows. Reading: the page clamps the fp32
    probability at 1e-30 before the log; in float64 LSE form that clamp never binds for
    |logit| well below 69, which holds for every workload here, so it is left out.
    """
    x = _f64(logits)
    t = np.asarray(targets).reshape(-1)
    n = x.shape[0]
    mx = x.max(axis=1)
    lse = mx + np.log(np.exp(x - mx[:, None]).sum(axis=1))
    return float((lse - x[np.arange(n), t]).sum() / n), lse


def softmax_ce_bwd(logits, targets, lse, dloss=1.0):
    """dlogits = (dloss / n) (softmax(row) - onehot(target)).

    [LM1] "Ops..." SoftmaxCrossEntropy backward: probability minus one at the target,
    scaled by the upstream gradient over the number of rows.
    """
    x = _f64(logits)
    t = np.asarray(targets).reshape(-1)
    n = x.shape[0]
    d = np.exp(x - _f64(lse)[:, None])
    d[np.arange(n), t] -= 1.0
    return d * (float(dloss) / n)


def softmax(x, temperature=1.0):
    """Row softmax of x / temperature, max subtracted first ([LM1] Softmax helper)."""
    z = _f64(x) / temperature
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


# -------------------------------------------------------------------------- AdamW
def adamw(p, g, m, v, t, lr, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0):
    """One AdamW update of one tensor at step t (t counts from 1). Returns (p, m, v).

    [LM1] "The optimizer: from gradient to step", AdamW listing (Loshchilov & Hutter):
    m = b1 m + (1 - b1) g; v = b2 v + (1 - b2) g^2; bias corrections 1 - b^t;
    p -= lr (mhat / (sqrt(vhat) + eps) + wd p), with the decay term using p before the
    update. The caller passes wd = 0 for tensors with fewer than two dimensions.
    """
    p, g, m, v = _f64(p), _f64(g), _f64(m), _f64(v)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    mhat = m / (1.0 - beta1 ** t)
    vhat = v / (1.0 - beta2 ** t)
    return p - lr * (mhat / (np.sqrt(vhat) + eps) + wd * p), m, v


# ------------------------------------------------------------------- generic ops, SGD
def add_fwd(a, b):
    """a + b with b broadcast over a's leading dimensions (b's shape is a's trailing shape).

    [LM1] "Ops..." op table: Add, with broadcast (a bias added to every row).
    """
    return _f64(a) + _f64(b)


def add_bwd(g, b_shape):
    """Contributions (da, db) of Add: da = g; db = g summed over the broadcast (leading)
    dimensions, so that it has b's shape. The reading of the broadcast rule: every row used
    b once, so b's gradient collects every row's."""
    g = _f64(g)
    lead = g.ndim - len(b_shape)
    return g.copy(), g.sum(axis=tuple(range(lead))).reshape(b_shape)


def mul_fwd(a, b):
    """Elementwise product. [LM1] "Ops...", Mul listing."""
    return _f64(a) * _f64(b)


def mul_bwd(a, b, g):
    """Mul's backward rule ([LM1] Mul listing): da += g b, db += g a."""
    g = _f64(g)
    return g * _f64(b), g * _f64(a)


def scale_fwd(a, s):
    """s a for a scalar s. [LM1] "Ops..." op table: Scale."""
    return float(s) * _f64(a)


def scale_bwd(s, g):
    """Scale's backward: da += s g."""
    return float(s) * _f64(g)


def sum_fwd(a):
    """The sum of every element (a scalar). [LM1] "Ops..." op table: Sum."""
    return float(np.sum(_f64(a)))


def sum_bwd(a_shape, g):
    """Sum's backward: every element of a receives the scalar upstream gradient g."""
    return np.full(a_shape, float(g), dtype=F64)


def tanh_fwd(x):
    """tanh elementwise. [LM1] "Ops..." op table: Tanh; [AD] Step 5 (the tanh neuron)."""
    return np.tanh(_f64(x))


def tanh_bwd(y, g):
    """Tanh's backward from its output y = tanh(x): dx += g (1 - y^2) ([AD] Step 5)."""
    y = _f64(y)
    return _f64(g) * (1.0 - y * y)


def sgd(p, g, lr):
    """Plain SGD: p - lr g. [LM1] "The optimizer: from gradient to step", Sgd listing."""
    return _f64(p) - float(lr) * _f64(g)
