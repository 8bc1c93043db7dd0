"""Oracle GPT-2-style decoder: training step (forward, backward, AdamW) and KV-cache decode.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the product path.

Model, as [LM4] "Loading weights into our classes" and "Generation with a KV cache"
describe it (the page with the model's own source is not available, so the block
structure is the reading below, pinned by the parameter count the pages print):

  x = wte[ids] + wpe[pos]
  for each layer: x += c_proj(attn(c_attn(ln_1(x))));  x += mlp_proj(gelu(c_fc(ln_2(x))))
  logits = ln_f(x) @ wte^T      (weight tying, MatMulT)

Every Linear has a bias and stores its weight [in, out]; the MLP widens 4x. With these,
the parameter count V*C + T*C + L*(12 C^2 + 13 C) + 2 C gives 124,439,808 for GPT-2
(V=50257, T=1024, C=768, L=12) and 457,440 for the pages' tiny model (V=39, T=64, C=96,
L=4), both of which the pages print.

Parameters are a dict keyed by the GPT-2 checkpoint names ([LM4] loading output).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import ops, sampling


@dataclass(frozen=True)
class Shape:
    V: int
    T: int
    C: int
    H: int
    L: int


def expected_shapes(s: Shape):
    """name -> shape of every parameter, 12 per layer plus 4 (148 for 12 layers)."""
    C = s.C
    out = {"wte.weight": (s.V, C), "wpe.weight": (s.T, C),
           "ln_f.weight": (C,), "ln_f.bias": (C,)}
    for i in range(s.L):
        p = f"h.{i}."
        out.update({
            p + "ln_1.weight": (C,), p + "ln_1.bias": (C,),
            p + "attn.c_attn.weight": (C, 3 * C), p + "attn.c_attn.bias": (3 * C,),
            p + "attn.c_proj.weight": (C, C), p + "attn.c_proj.bias": (C,),
            p + "ln_2.weight": (C,), p + "ln_2.bias": (C,),
            p + "mlp.c_fc.weight": (C, 4 * C), p + "mlp.c_fc.bias": (4 * C,),
            p + "mlp.c_proj.weight": (4 * C, C), p + "mlp.c_proj.bias": (C,),
        })
    return out


def param_count(s: Shape) -> int:
    return int(sum(np.prod(v) for v in expected_shapes(s).values()))


def check_params(params, s: Shape):
    """Raise on a missing tensor or a shape mismatch ([LM4] loading throws on mismatch)."""
    exp = expected_shapes(s)
    for name, shape in exp.items():
        if name not in params:
            raise KeyError(name)
        if tuple(params[name].shape) != shape:
            raise ValueError(f"{name}: {params[name].shape} vs {shape}")


def _w(params, name):
    return np.asarray(params[name], dtype=np.float64)


# ------------------------------------------------------------------ training step
def forward(params, ids, s: Shape):
    """Logits [B, T, V] and the saved activations for backward."""
    ids = np.asarray(ids)
    B, T = ids.shape
    N = B * T
    C = s.C
    act = {"ids": ids, "layers": []}
    x = ops.embedding_fwd(ids, params["wte.weight"], params["wpe.weight"]).reshape(N, C)
    for i in range(s.L):
        p = f"h.{i}."
        a = {"x_in": x}
        a["ln1"], a["mu1"], a["rs1"] = ops.layernorm_fwd(x, _w(params, p + "ln_1.weight"),
                                                         _w(params, p + "ln_1.bias"))
        qkv = ops.matmul_fwd(a["ln1"], _w(params, p + "attn.c_attn.weight")) \
            + _w(params, p + "attn.c_attn.bias")
        a["qkv"] = qkv
        y, a["P"], a["lse"] = ops.attention_fwd(qkv.reshape(B, T, 3 * C), s.H)
        a["y"] = y.reshape(N, C)
        x = x + ops.matmul_fwd(a["y"], _w(params, p + "attn.c_proj.weight")) \
            + _w(params, p + "attn.c_proj.bias")
        a["x_mid"] = x
        a["ln2"], a["mu2"], a["rs2"] = ops.layernorm_fwd(x, _w(params, p + "ln_2.weight"),
                                                         _w(params, p + "ln_2.bias"))
        a["pre"] = ops.matmul_fwd(a["ln2"], _w(params, p + "mlp.c_fc.weight")) \
            + _w(params, p + "mlp.c_fc.bias")
        a["h"] = ops.gelu_fwd(a["pre"])
        x = x + ops.matmul_fwd(a["h"], _w(params, p + "mlp.c_proj.weight")) \
            + _w(params, p + "mlp.c_proj.bias")
        act["layers"].append(a)
    act["x_out"] = x
    act["lnf"], act["muf"], act["rsf"] = ops.layernorm_fwd(x, _w(params, "ln_f.weight"),
                                                          _w(params, "ln_f.bias"))
    logits = ops.matmul_t_fwd(act["lnf"], _w(params, "wte.weight"))
    return logits.reshape(B, T, s.V), act


def backward(params, act, dlogits, s: Shape):
    """Gradients of every parameter (float64 dict) given dlogits [N, V].

    Reverse order of forward; the residual stream's gradient is the sum of the skip path
    and the branch path ([LM1] "Why += and not =": a tensor used twice adds both parts).
    The embedding gradient here is accumulated in float64 (embedding_bwd in ops is the
    float32 ordered definition used for the exact single-op comparison).
    """
    ids = act["ids"]
    B, T = ids.shape
    N, C = B * T, s.C
    grads = {k: np.zeros(v.shape, dtype=np.float64) for k, v in params.items()}
    dlogits = np.asarray(dlogits, dtype=np.float64).reshape(N, s.V)
    dlnf, dwte = ops.matmul_t_bwd(act["lnf"], _w(params, "wte.weight"), dlogits)
    grads["wte.weight"] += dwte
    dx, dg, db = ops.layernorm_bwd(act["x_out"], _w(params, "ln_f.weight"), act["muf"],
                                   act["rsf"], dlnf)
    grads["ln_f.weight"] += dg
    grads["ln_f.bias"] += db
    for i in reversed(range(s.L)):
        p = f"h.{i}."
        a = act["layers"][i]
        # x = x_mid + h @ Wp + bp
        dh, dWp = ops.matmul_bwd(a["h"], _w(params, p + "mlp.c_proj.weight"), dx)
        grads[p + "mlp.c_proj.weight"] += dWp
        grads[p + "mlp.c_proj.bias"] += ops.bias_bwd(dx)
        dpre = ops.gelu_bwd(a["pre"], dh)
        dln2, dWfc = ops.matmul_bwd(a["ln2"], _w(params, p + "mlp.c_fc.weight"), dpre)
        grads[p + "mlp.c_fc.weight"] += dWfc
        grads[p + "mlp.c_fc.bias"] += ops.bias_bwd(dpre)
        d, dg, db = ops.layernorm_bwd(a["x_mid"], _w(params, p + "ln_2.weight"), a["mu2"],
                                      a["rs2"], dln2)
        grads[p + "ln_2.weight"] += dg
        grads[p + "ln_2.bias"] += db
        dx = dx + d
        # x_mid = x_in + y @ Wo + bo
        dy, dWo = ops.matmul_bwd(a["y"], _w(params, p + "attn.c_proj.weight"), dx)
        grads[p + "attn.c_proj.weight"] += dWo
        grads[p + "attn.c_proj.bias"] += ops.bias_bwd(dx)
        dqkv = ops.attention_bwd(a["qkv"].reshape(B, T, 3 * C), a["P"],
                                 dy.reshape(B, T, C), s.H).reshape(N, 3 * C)
        dln1, dWqkv = ops.matmul_bwd(a["ln1"], _w(params, p + "attn.c_attn.weight"), dqkv)
        grads[p + "attn.c_attn.weight"] += dWqkv
        grads[p + "attn.c_attn.bias"] += ops.bias_bwd(dqkv)
        d, dg, db = ops.layernorm_bwd(a["x_in"], _w(params, p + "ln_1.weight"), a["mu1"],
                                      a["rs1"], dln1)
        grads[p + "ln_1.weight"] += dg
        grads[p + "ln_1.bias"] += db
        dx = dx + d
    flat = ids.reshape(-1)
    np.add.at(grads["wte.weight"], flat, dx)
    np.add.at(grads["wpe.weight"], np.arange(N) % T, dx)
    return grads


def loss_and_grads(params, ids, targets, s: Shape):
    """(loss, grads, logits [N, V], lse [N]) of one batch, dloss = 1."""
    check_params(params, s)
    logits, act = forward(params, ids, s)
    B, T = np.asarray(ids).shape
    logits = logits.reshape(B * T, s.V)
    loss, lse = ops.softmax_ce_fwd(logits, targets)
    dlogits = ops.softmax_ce_bwd(logits, targets, lse, 1.0)
    return loss, backward(params, act, dlogits, s), logits, lse


def adamw_step(params, grads, state, t, lr, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0):
    """AdamW over every tensor; weight decay only on tensors with two or more dims.

    [LM1] "The optimizer: from gradient to step": vectors (biases, LayerNorm gains) are not
    decayed. state maps name -> (m, v); returns (new params, new state), all float64.
    """
    new_p, new_s = {}, {}
    for name, p in params.items():
        m, v = state.get(name, (np.zeros(p.shape), np.zeros(p.shape)))
        w = wd if np.ndim(p) >= 2 else 0.0
        new_p[name], mm, vv = ops.adamw(p, grads[name], m, v, t, lr, beta1, beta2, eps, w)
        new_s[name] = (mm, vv)
    return new_p, new_s


# ------------------------------------------------------------------- KV-cache decode
class KvCache:
    """Keys and values of every position seen so far, per layer: [B, H, Tmax, hs] each.

    [LM4] "Generation with a KV cache" (one key and one value row of C numbers per layer per
    position, appended as positions arrive).
    """

    def __init__(self, s: Shape, B: int, Tmax: int):
        hs = s.C // s.H
        self.k = [np.zeros((B, s.H, Tmax, hs)) for _ in range(s.L)]
        self.v = [np.zeros((B, s.H, Tmax, hs)) for _ in range(s.L)]
        self.length = 0


def decode_step(params, cache: KvCache, tokens, pos: int, s: Shape):
    """Logits [B, V] for one new token per row at position `pos`, appending to the cache.

    [LM4] "Generation with a KV cache": the token's row through every layer with that
    layer's cache; attention over every cached position j <= pos needs no mask because the
    cache holds only the past; then ln_f and the tied head.
    """
    tokens = np.asarray(tokens).reshape(-1)
    B = tokens.shape[0]
    C, H = s.C, s.H
    hs = C // H
    if pos >= cache.k[0].shape[2]:
        raise IndexError("KV cache full")
    x = _w(params, "wte.weight")[tokens] + _w(params, "wpe.weight")[pos]
    for i in range(s.L):
        p = f"h.{i}."
        h1, _, _ = ops.layernorm_fwd(x, _w(params, p + "ln_1.weight"), _w(params, p + "ln_1.bias"))
        qkv = h1 @ _w(params, p + "attn.c_attn.weight") + _w(params, p + "attn.c_attn.bias")
        q = qkv[:, :C].reshape(B, H, hs)
        cache.k[i][:, :, pos] = qkv[:, C:2 * C].reshape(B, H, hs)
        cache.v[i][:, :, pos] = qkv[:, 2 * C:].reshape(B, H, hs)
        K = cache.k[i][:, :, :pos + 1]
        Vv = cache.v[i][:, :, :pos + 1]
        sc = np.einsum("bhd,bhjd->bhj", q, K) / np.sqrt(hs)
        pr = ops.softmax(sc)
        y = np.einsum("bhj,bhjd->bhd", pr, Vv).reshape(B, C)
        x = x + y @ _w(params, p + "attn.c_proj.weight") + _w(params, p + "attn.c_proj.bias")
        h2, _, _ = ops.layernorm_fwd(x, _w(params, p + "ln_2.weight"), _w(params, p + "ln_2.bias"))
        m = ops.gelu_fwd(h2 @ _w(params, p + "mlp.c_fc.weight") + _w(params, p + "mlp.c_fc.bias"))
        x = x + m @ _w(params, p + "mlp.c_proj.weight") + _w(params, p + "mlp.c_proj.bias")
    cache.length = pos + 1
    hf, _, _ = ops.layernorm_fwd(x, _w(params, "ln_f.weight"), _w(params, "ln_f.bias"))
    return hf @ _w(params, "wte.weight").T


def prefill(params, prompt, s: Shape, Tmax: int):
    """Fill a fresh cache with a [B, Tp] prompt; return (cache, logits of the last position).

    The pages feed the prompt one token at a time through decode_step; one causal forward
    over the whole prompt is the same arithmetic ([LM4] "Generation with a KV cache": the
    cached step is the same math as the full forward), and is what this does.
    """
    prompt = np.asarray(prompt)
    B, Tp = prompt.shape
    C, H = s.C, s.H
    cache = KvCache(s, B, Tmax)
    N = B * Tp
    x = ops.embedding_fwd(prompt, params["wte.weight"], params["wpe.weight"]).reshape(N, C)
    for i in range(s.L):
        p = f"h.{i}."
        h1, _, _ = ops.layernorm_fwd(x, _w(params, p + "ln_1.weight"), _w(params, p + "ln_1.bias"))
        qkv = h1 @ _w(params, p + "attn.c_attn.weight") + _w(params, p + "attn.c_attn.bias")
        q3 = qkv.reshape(B, Tp, 3 * C)
        cache.k[i][:, :, :Tp] = ops.split_heads(q3[..., C:2 * C], H)
        cache.v[i][:, :, :Tp] = ops.split_heads(q3[..., 2 * C:], H)
        y, _, _ = ops.attention_fwd(q3, H)
        x = x + y.reshape(N, C) @ _w(params, p + "attn.c_proj.weight") \
            + _w(params, p + "attn.c_proj.bias")
        h2, _, _ = ops.layernorm_fwd(x, _w(params, p + "ln_2.weight"), _w(params, p + "ln_2.bias"))
        m = ops.gelu_fwd(h2 @ _w(params, p + "mlp.c_fc.weight") + _w(params, p + "mlp.c_fc.bias"))
        x = x + m @ _w(params, p + "mlp.c_proj.weight") + _w(params, p + "mlp.c_proj.bias")
    cache.length = Tp
    last = x.reshape(B, Tp, C)[:, -1]
    hf, _, _ = ops.layernorm_fwd(last, _w(params, "ln_f.weight"), _w(params, "ln_f.bias"))
    return cache, hf @ _w(params, "wte.weight").T


def generate(params, prompt, n_steps: int, s: Shape, top_k=0, temperature=1.0, seed=0,
             counter0=0, forced=None):
    """Cached generation: prefill, then n_steps decode steps of select-and-feed-back.

    The prefill's last logits give selection 0; decode step i (position Tp + i) consumes
    selection i and gives the logits of selection i + 1, so there are n_steps + 1
    selections and the cache ends holding Tp + n_steps positions. Selection is greedy when
    top_k == 1 or temperature == 0, else top-k sampling with the Philox draw of step
    counter0 + i. If `forced` ([n_steps, B] ids) is given, those ids are fed back instead
    of the selected ones (teacher forcing); selections and logits are still recorded.
    Returns (selected [n_steps + 1, B], logits [n_steps + 1, B, V]).
    """
    prompt = np.asarray(prompt)
    B, Tp = prompt.shape
    cache, logits = prefill(params, prompt, s, Tp + n_steps)
    picks, all_logits = [], []
    for i in range(n_steps + 1):
        all_logits.append(logits)
        if top_k == 1 or temperature == 0:
            nxt = sampling.greedy(logits)
        else:
            nxt = np.array([sampling.topk_sample(logits[b], top_k, temperature,
                                                 sampling.uniform(seed, counter0 + i, b))
                            for b in range(B)], dtype=np.int32)
        picks.append(nxt)
        if i < n_steps:
            feed = nxt if forced is None else np.asarray(forced[i])
            logits = decode_step(params, cache, feed, Tp + i, s)
    return np.array(picks), np.array(all_logits)
