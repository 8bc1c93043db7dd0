"""Seeded synthetic inputs for the decoder-step library, its tests and its bench.

This module holds no arithmetic of the decoder step itself. It only turns a seed into
random numbers (SplitMix64, Steele, Lea & Flood, "Fast Splittable Pseudorandom Number
Generators", OOPSLA 2014), and those numbers into the inputs the workloads describe:

* token ids uniform in [0, V), drawn as B x (T+1) so that the inputs are ids[:, :T] and the
  next-token targets are ids[:, 1:];
* weights of every parameter tensor with two or more dimensions ~ N(0, 0.02), biases 0,
  LayerNorm gains 1 and LayerNorm biases 0;
* N(0, 1) operands for single-op checks.

Both the oracle's callers and the CUDA path's callers draw from here, so the two sides see
bit-identical inputs; neither side imports the other.
"""
from __future__ import annotations

import math
import os
from collections import OrderedDict
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _parallel_chunks(n: int, fn) -> None:
    """Run fn(s, e) over [0, n) in chunks; numpy releases the GIL inside each chunk."""
    spans = [(s, min(n, s + _CHUNK)) for s in range(0, n, _CHUNK)]
    if len(spans) <= 1:
        for s, e in spans:
            fn(s, e)
        return
    with ThreadPoolExecutor(max_workers=min(len(spans), os.cpu_count() or 1)) as pool:
        list(pool.map(lambda se: fn(*se), spans))


class Stream:
    """A SplitMix64 sequence: output i is mix(seed + (i + 1) * golden_gamma)."""

    def __init__(self, seed: int):
        self.seed = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
        self.counter = 0

    def _u64_at(self, start: int, n: int) -> np.ndarray:
        with np.errstate(over="ignore"):
            idx = np.arange(start + 1, start + n + 1, dtype=np.uint64)
            return _mix64(self.seed + idx * _GAMMA)

    def u64(self, n: int) -> np.ndarray:
        out = np.empty(n, dtype=np.uint64)
        base = self.counter

        def fill(s, e):
            out[s:e] = self._u64_at(base + s, e - s)

        _parallel_chunks(n, fill)
        self.counter += n
        return out

    def uniform(self, n: int) -> np.ndarray:
        """Uniform doubles in [0, 1) from the top 53 bits."""
        return (self.u64(n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)

    def ints(self, n: int, hi: int) -> np.ndarray:
        """Integers uniform in [0, hi) as int32 (floor(u * hi))."""
        return np.floor(self.uniform(n) * hi).astype(np.int32)

    def normal(self, n: int, std: float = 1.0) -> np.ndarray:
        """N(0, std^2) as float32, Box-Muller (cosine branch) on pairs of uniforms."""
        out = np.empty(n, dtype=np.float32)
        base = self.counter

        def fill(s, e):
            u = (self._u64_at(base + 2 * s, 2 * (e - s)) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
            r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
            out[s:e] = (r * np.cos(2.0 * math.pi * u[1::2]) * std).astype(np.float32)

        _parallel_chunks(n, fill)
        self.counter += 2 * n
        return out


@dataclass(frozen=True)
class GptShape:
    """Sizes of a GPT-2-style decoder: vocabulary, context, width, heads, layers."""

    V: int
    T: int
    C: int
    H: int
    L: int

    @property
    def hs(self) -> int:
        return self.C // self.H


# The tiny character-level model and the GPT-2-124M shape the workloads name.
TINY = GptShape(V=64, T=64, C=96, H=4, L=4)
GPT2_124M = GptShape(V=50257, T=1024, C=768, H=12, L=12)


def param_names_shapes(s: GptShape):
    """Names and shapes of the parameter tensors, in the GPT-2 checkpoint naming."""
    C = s.C
    out = [("wte.weight", (s.V, C)), ("wpe.weight", (s.T, C))]
    for i in range(s.L):
        p = f"h.{i}."
        out += [
            (p + "ln_1.weight", (C,)), (p + "ln_1.bias", (C,)),
            (p + "attn.c_attn.weight", (C, 3 * C)), (p + "attn.c_attn.bias", (3 * C,)),
            (p + "attn.c_proj.weight", (C, C)), (p + "attn.c_proj.bias", (C,)),
            (p + "ln_2.weight", (C,)), (p + "ln_2.bias", (C,)),
            (p + "mlp.c_fc.weight", (C, 4 * C)), (p + "mlp.c_fc.bias", (4 * C,)),
            (p + "mlp.c_proj.weight", (4 * C, C)), (p + "mlp.c_proj.bias", (C,)),
        ]
    out += [("ln_f.weight", (C,)), ("ln_f.bias", (C,))]
    return out


def gpt_params(s: GptShape, stream: Stream, std: float = 0.02) -> "OrderedDict[str, np.ndarray]":
    """Initial parameters: matrices N(0, std^2), biases 0, LayerNorm gains 1 (float32)."""
    params = OrderedDict()
    for name, shape in param_names_shapes(s):
        n = int(np.prod(shape))
        if len(shape) >= 2:
            params[name] = stream.normal(n, std).reshape(shape)
        elif name.endswith("ln_1.weight") or name.endswith("ln_2.weight") or name == "ln_f.weight":
            params[name] = np.ones(shape, dtype=np.float32)
        else:
            params[name] = np.zeros(shape, dtype=np.float32)
    return params


def token_batch(s: GptShape, B: int, stream: Stream, T: int | None = None):
    """(inputs [B,T], targets [B,T]) int32: B x (T+1) uniform ids, shifted by one."""
    T = s.T if T is None else T
    ids = stream.ints(B * (T + 1), s.V).reshape(B, T + 1)
    return np.ascontiguousarray(ids[:, :T]), np.ascontiguousarray(ids[:, 1:])


def training_case(s: GptShape, B: int, seed: int, T: int | None = None):
    """The seeded training-step workload: ids first, then the parameters."""
    st = Stream(seed)
    ids, targets = token_batch(s, B, st, T)
    params = gpt_params(s, st)
    return ids, targets, params


def prompt_case(s: GptShape, B: int, Tp: int, seed: int):
    """The seeded decode workload: a [B, Tp] prompt of uniform ids, then the parameters."""
    st = Stream(seed)
    prompt = st.ints(B * Tp, s.V).reshape(B, Tp)
    params = gpt_params(s, st)
    return prompt, params


def circle_case(seed: int, n: int = 256, hidden: int = 16):
    """The circle task's seeded inputs: n points uniform in [-1, 1)^2 (float32 [n, 2]), label 1
    inside the circle x^2 + y^2 < 0.5 else 0 (int32 [n]), and the 2 -> hidden -> 2 network's
    initial weights: N(0, 0.5^2) matrices [in, out], zero biases."""
    st = Stream(seed)
    xs = (st.uniform(2 * n) * 2.0 - 1.0).astype(np.float32).reshape(n, 2)
    x64 = xs.astype(np.float64)
    ys = ((x64[:, 0] ** 2 + x64[:, 1] ** 2) < 0.5).astype(np.int32)
    w1 = st.normal(2 * hidden, 0.5).reshape(2, hidden)
    w2 = st.normal(hidden * 2, 0.5).reshape(hidden, 2)
    return xs, ys, (w1, np.zeros(hidden, np.float32), w2, np.zeros(2, np.float32))


def xor_case(seed: int, hidden: int = 4):
    """XOR's four points (float32 [4, 2]), targets -1 / 1 (float32 [4, 1]) and the [2, hidden, 1]
    network's initial weights: uniform in [-1, 1) matrices [in, out], zero biases."""
    st = Stream(seed)
    xs = np.array([[0, 0], [0, 1], [1, 0], [1, 1]], np.float32)
    ys = np.array([[-1], [1], [1], [-1]], np.float32)
    w1 = (st.uniform(2 * hidden) * 2.0 - 1.0).astype(np.float32).reshape(2, hidden)
    w2 = (st.uniform(hidden) * 2.0 - 1.0).astype(np.float32).reshape(hidden, 1)
    return xs, ys, (w1, np.zeros(hidden, np.float32), w2, np.zeros(1, np.float32))
