"""Pins of the oracle's model, decode and sampling: the pages' printed sizes, whole-model
finite differences, the cached-vs-full invariant, published Philox vectors."""
import math
import os

import numpy as np
import pytest

import synth
from oracle import gpt, ops, sampling
from tests.conftest import GOLDEN


def _shape(s):
    return gpt.Shape(V=s.V, T=s.T, C=s.C, H=s.H, L=s.L)


def test_parameter_counts_match_the_pages(page):
    g2 = gpt.Shape(V=50257, T=1024, C=768, H=12, L=12)
    assert gpt.param_count(g2) == page["gpt2.params"]
    assert len(gpt.expected_shapes(g2)) == page["gpt2.tensors"]
    assert np.prod(gpt.expected_shapes(g2)["wte.weight"]) == page["gpt2.wte_numbers"]
    tiny = gpt.Shape(V=int(page["tiny.vocab"]), T=64, C=96, H=4, L=4)
    assert gpt.param_count(tiny) == page["tiny.params"]
    # "about 85 million" multiply-adds per token in the layers: 12 C^2 per layer
    macs = 12 * 12 * 768 ** 2
    assert abs(macs - page["gpt2.block_macs_per_token_approx"]) / macs < 0.01
    # the synthetic generator produces exactly the oracle's parameter set
    names = dict(synth.param_names_shapes(synth.GPT2_124M))
    assert names == {k: tuple(v) for k, v in gpt.expected_shapes(g2).items()}


def test_shape_mismatch_raises():
    s = gpt.Shape(V=5, T=4, C=8, H=2, L=1)
    params = {k: np.zeros(v) for k, v in gpt.expected_shapes(s).items()}
    params["h.0.attn.c_attn.weight"] = np.zeros((24, 8))  # transposed
    with pytest.raises(ValueError):
        gpt.check_params(params, s)


MINI = synth.GptShape(V=7, T=4, C=8, H=2, L=2)


def _mini_case(seed=3, B=2):
    ids, targets, params = synth.training_case(MINI, B, seed)
    st = synth.Stream(seed + 100)
    # perturb biases and gains away from 0 / 1 so their gradients are exercised fully
    p64 = {}
    for k, v in params.items():
        v = v.astype(np.float64)
        if v.ndim == 1:
            v = v + st.normal(v.size, 0.3).astype(np.float64)
        else:
            v = v * 10  # std 0.2, so attention and GELU leave their linear regimes
        p64[k] = v
    return ids, targets, p64


def test_whole_model_gradient_check():
    ids, targets, params = _mini_case()
    s = _shape(MINI)
    loss, grads, _, _ = gpt.loss_and_grads(params, ids, targets, s)
    h = 1e-6
    worst = 0.0
    for name, p in params.items():
        num = np.zeros_like(p)
        for i in np.ndindex(p.shape):
            old = p[i]
            p[i] = old + h
            lp = gpt.loss_and_grads(params, ids, targets, s)[0]
            p[i] = old - h
            lm = gpt.loss_and_grads(params, ids, targets, s)[0]
            p[i] = old
            num[i] = (lp - lm) / (2 * h)
        a = grads[name]
        rel = np.linalg.norm(a - num) / (np.linalg.norm(a) + np.linalg.norm(num))
        worst = max(worst, rel)
        assert rel < 1e-6, name
    assert worst < 1e-6


def test_initial_loss_is_near_log_vocab():
    ids, targets, params = synth.training_case(synth.TINY, 8, 0)
    loss, _, _, _ = gpt.loss_and_grads(params, ids, targets, _shape(synth.TINY))
    assert abs(loss - math.log(64)) < 0.05


def test_adamw_step_decays_only_matrices():
    ids, targets, params = _mini_case()
    s = _shape(MINI)
    grads = {k: np.zeros_like(v) for k, v in params.items()}
    newp, _ = gpt.adamw_step(params, grads, {}, 1, lr=0.1, wd=0.5)
    for k, v in params.items():
        if v.ndim >= 2:
            np.testing.assert_allclose(newp[k], v * (1 - 0.05), rtol=1e-15)
        else:
            np.testing.assert_array_equal(newp[k], v)


def test_cached_decode_equals_full_forward(page):
    s = gpt.Shape(V=11, T=12, C=8, H=2, L=2)
    st = synth.Stream(9)
    prompt = st.ints(2 * 3, s.V).reshape(2, 3)
    params = {k: v.astype(np.float64) * (5 if v.ndim > 1 else 1)
              for k, v in synth.gpt_params(synth.GptShape(**s.__dict__), st).items()}
    forced = st.ints(2 * 6, s.V).reshape(6, 2)
    picks, logits = gpt.generate(params, prompt, 6, s, top_k=1, forced=forced)
    full_ids = np.concatenate([prompt, forced.T], axis=1)
    full, _ = gpt.forward(params, full_ids, s)
    for i in range(7):
        np.testing.assert_allclose(logits[i], full[:, 2 + i], rtol=0, atol=1e-12)
    assert np.abs(logits[0] - full[:, 2]).max() < page["kv_vs_full.max_abs"]
    np.testing.assert_array_equal(picks, np.argmax(logits, axis=-1))
    # a token-by-token prompt (the pages' way) gives the same cache and logits
    cache = gpt.KvCache(s, 2, 9)
    for t in range(3):
        step_logits = gpt.decode_step(params, cache, prompt[:, t], t, s)
    np.testing.assert_allclose(step_logits, logits[0], atol=1e-12)
    with pytest.raises(IndexError):
        gpt.decode_step(params, gpt.KvCache(s, 2, 1), prompt[:, 0], 1, s)


def test_philox_known_answers():
    with open(os.path.join(GOLDEN, "philox4x32_10_kat.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for r in rows:
        w = [int(x, 16) for x in r]
        assert sampling.philox4x32_10(w[0:4], w[4:6]) == tuple(w[6:10])


def test_uniform_draws_are_in_range_and_distinct():
    us = [sampling.uniform(4, step, row) for step in range(64) for row in range(16)]
    assert all(0.0 <= u < 1.0 for u in us)
    assert len(set(us)) > 1000
    assert abs(np.mean(us) - 0.5) < 0.03


def test_topk_keeps_ties_and_greedy_takes_lowest_index():
    row = np.array([0.5, 2.0, 1.0, 2.0, 1.0, 1.0, -3.0])
    np.testing.assert_array_equal(sampling.topk_keep(row, 3), row >= 1.0)  # 3rd largest is 1.0
    assert sampling.topk_keep(row, 3).sum() == 5
    assert sampling.topk_keep(row, 0).all() and sampling.topk_keep(row, 7).all()
    assert sampling.greedy(row) == 1
    # u = 0 takes the first kept index; u just below 1 the last kept index
    assert sampling.topk_sample(row, 2, 1.0, 0.0) == 1
    assert sampling.topk_sample(row, 2, 1.0, 1 - 2 ** -24) == 3
    # k = 1 with a unique maximum is greedy for any u
    r2 = np.array([0.1, 0.3, 0.2])
    assert all(sampling.topk_sample(r2, 1, 1.0, u) == 1 for u in (0.0, 0.5, 0.999))
    # empirical frequencies follow the temperature softmax of the kept set
    r3 = np.array([1.0, 0.0, 2.0, -1.0])
    counts = np.zeros(4)
    for step in range(4000):
        counts[sampling.topk_sample(r3, 3, 0.5, sampling.uniform(7, step, 0))] += 1
    p = np.exp(np.array([1.0, 0.0, 2.0]) / 0.5)
    p /= p.sum()
    np.testing.assert_allclose(counts[:3] / 4000, p, atol=0.03)
    assert counts[3] == 0
