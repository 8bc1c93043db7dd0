"""Python binding of libgk: the same entry points as include/gk.h, argument marshalling only.

Tensor arguments accept a torch tensor (its data_ptr is passed), a raw integer address or
None (NULL). Every computation runs in libgk's CUDA kernels; there is no fallback: importing
this module raises if libgk.so has not been built for this machine.
"""
from __future__ import annotations

import ctypes as ct
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgk.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
_lib = ct.CDLL(LIB_PATH)

# status codes and enums (include/gk.h)
GK_OK, GK_ERR_ARG, GK_ERR_ALIGN, GK_ERR_UNSUPPORTED, GK_ERR_CUDA, GK_ERR_TIMEOUT, GK_ERR_OVERFLOW, GK_ERR_INDEX, \
    GK_ERR_WORKSPACE, GK_ERR_IO, GK_ERR_FORMAT = range(11)
GK_F32, GK_BF16, GK_BF16X2 = 0, 1, 2
GK_MATH_FP32, GK_MATH_3XTF32 = 0, 1
GK_ACT_NONE, GK_ACT_GELU = 0, 1
(GK_T_WTE, GK_T_WPE, GK_T_LN1_W, GK_T_LN1_B, GK_T_ATTN_W, GK_T_ATTN_B, GK_T_ATTNPROJ_W, GK_T_ATTNPROJ_B,
 GK_T_LN2_W, GK_T_LN2_B, GK_T_FC_W, GK_T_FC_B, GK_T_MLPPROJ_W, GK_T_MLPPROJ_B, GK_T_LNF_W, GK_T_LNF_B) = range(16)

STATUS_NAMES = {0: "GK_OK", 1: "GK_ERR_ARG", 2: "GK_ERR_ALIGN", 3: "GK_ERR_UNSUPPORTED", 4: "GK_ERR_CUDA",
                5: "GK_ERR_TIMEOUT", 6: "GK_ERR_OVERFLOW", 7: "GK_ERR_INDEX", 8: "GK_ERR_WORKSPACE", 9: "GK_ERR_IO",
                10: "GK_ERR_FORMAT"}

P = ct.c_void_p
I32, I64, F32 = ct.c_int, ct.c_int64, ct.c_float


class GkError(RuntimeError):
    def __init__(self, status, where, msg):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class gk_param(ct.Structure):
    _fields_ = [("p", P), ("g", P), ("m", P), ("v", P), ("n", I64), ("decay", I32), ("p_bf16", P), ("p_bf16_lo", P)]


class gk_gpt_cfg(ct.Structure):
    _fields_ = [("V", I32), ("T", I32), ("C", I32), ("H", I32), ("L", I32)]


class gk_sample_cfg(ct.Structure):
    _fields_ = [("top_k", I32), ("temperature", F32), ("seed", ct.c_uint64), ("counter", ct.c_uint64)]


_SIGS = {
    "gk_ctx_create": (I32, [ct.POINTER(P), P, ct.c_size_t]),
    "gk_ctx_destroy": (None, [P]),
    "gk_ctx_set_stream": (I32, [P, P]),
    "gk_set_math": (I32, [P, I32]),
    "gk_sync": (I32, [P]),
    "gk_last_error": (ct.c_char_p, [P]),
    "gk_launch_count": (I64, [P]),
    "gk_selftest_wait_timeout": (I32, [P, I64, I32, P]),
    "gk_embedding_fwd": (I32, [P, P, P, P, P, I32, I32, I32, I32]),
    "gk_embedding_bwd": (I32, [P, P, P, P, P, I32, I32, I32, I32]),
    "gk_layernorm_fwd": (I32, [P, P, P, P, P, I32, P, P, I64, I32, F32, P]),
    "gk_lmhead_ce_fwd": (I32, [P, I32, P, I64, P, I64, P, P, P, I64, I64, I64]),
    "gk_lmhead_ce_bwd": (I32, [P, I32, P, I64, P, I64, P, P, P, P, I64, I32, P, I64, P, I64, I64, I64, I64]),
    "gk_decode_run": (I32, [P, P, P, P, P, P, P, I32]),
    "gk_generate_uncached": (I32, [P, P, P, P, I32, I32, P, P]),
    "gk_add_fwd": (I32, [P, P, P, P, I64, I64]),
    "gk_add_bwd": (I32, [P, P, P, P, I64, I64, I32]),
    "gk_mul_fwd": (I32, [P, P, P, P, I64]),
    "gk_mul_bwd": (I32, [P, P, P, P, P, P, I64, I32]),
    "gk_scale_fwd": (I32, [P, P, F32, P, I64]),
    "gk_scale_bwd": (I32, [P, P, F32, P, I64, I32]),
    "gk_sum_fwd": (I32, [P, P, P, I64]),
    "gk_sum_bwd": (I32, [P, P, P, I64, I32]),
    "gk_tanh_fwd": (I32, [P, P, P, I64]),
    "gk_tanh_bwd": (I32, [P, P, P, P, I64, I32]),
    "gk_sgd_step": (I32, [P, P, P, I64, F32]),
    "gk_layernorm_bwd": (I32, [P, P, P, P, P, P, P, I32, P, P, P, P, I64, I32]),
    "gk_layernorm_bwd_noalloc": (I32, [P, P, P, P, P, P, P, I32, P, P, P, I64, I32]),
    "gk_gelu_fwd": (I32, [P, P, P, I64]),
    "gk_gelu_bwd": (I32, [P, P, P, P, I64]),
    "gk_matmul_fwd": (I32, [P, I32, P, I64, P, I64, I32, P, P, I64, P, I64, I32, I64, I64, I64, I32, P, I64, P, P]),
    "gk_matmul_bwd": (I32, [P, I32, P, I64, P, I64, I32, P, I64, P, I64, I32, I32, P, I64, P, I64, P, I64, I64,
                            I64]),
    "gk_attn_fwd": (I32, [P, I32, P, P, P, I32, I32, I32, I32]),
    "gk_attn_bwd": (I32, [P, I32, P, P, P, P, P, I32, I32, I32, I32]),
    "gk_softmax_ce_fwd": (I32, [P, P, I64, P, P, P, I64, I32]),
    "gk_softmax_ce_bwd": (I32, [P, P, I64, P, P, P, P, I64, I32, I64, I32]),
    "gk_to_bf16": (I32, [P, P, P, P, I64]),
    "gk_adamw_step": (I32, [P, ct.POINTER(gk_param), I32, F32, F32, F32, F32, F32, I32, I32]),
    "gk_gpt_offset": (I64, [ct.POINTER(gk_gpt_cfg), I32, I32]),
    "gk_gpt_numel": (I64, [ct.POINTER(gk_gpt_cfg)]),
    "gk_gpt_n_decay": (I64, [ct.POINTER(gk_gpt_cfg)]),
    "gk_kv_create": (I32, [P, ct.POINTER(P), ct.POINTER(gk_gpt_cfg), I32, I32]),
    "gk_kv_destroy": (None, [P]),
    "gk_kv_data": (P, [P]),
    "gk_kv_length": (I32, [P]),
    "gk_prefill": (I32, [P, P, P, P, I32, P]),
    "gk_decode_step": (I32, [P, P, P, P, P, P, ct.POINTER(gk_sample_cfg)]),
    "gk_sample": (I32, [P, P, P, I64, P, ct.POINTER(gk_sample_cfg)]),
    "gk_st_open": (I32, [ct.c_char_p, ct.POINTER(P)]),
    "gk_st_close": (None, [P]),
    "gk_st_count": (I32, [P]),
    "gk_st_name": (ct.c_char_p, [P, I32]),
    "gk_st_dtype": (ct.c_char_p, [P, I32]),
    "gk_st_ndim": (I32, [P, I32]),
    "gk_st_shape": (ct.POINTER(I64), [P, I32]),
    "gk_st_find": (I32, [P, ct.c_char_p]),
    "gk_st_metadata": (ct.c_char_p, [P, ct.c_char_p]),
    "gk_st_read_f32": (I32, [P, I32, P, I64, I32]),
    "gk_st_write_f32": (I32, [ct.c_char_p, I32, ct.POINTER(ct.c_char_p), ct.POINTER(I32), ct.POINTER(I64),
                              ct.POINTER(P), I32, I32, ct.POINTER(ct.c_char_p), ct.POINTER(ct.c_char_p)]),
    "gk_st_last_error": (ct.c_char_p, []),
}

EXPORTED = tuple(_SIGS)

for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def _p(x):
    """Address of a tensor / int / None for a pointer argument."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


class Ctx:
    """A libgk context bound to a CUDA stream (an int handle or a torch.cuda.Stream)."""

    def __init__(self, stream=0, workspace_bytes=64 << 20):
        h = P()
        s = stream if isinstance(stream, int) else stream.cuda_stream
        _check(None, _lib.gk_ctx_create(ct.byref(h), P(s), workspace_bytes), "gk_ctx_create")
        self.handle = h

    @property
    def _as_parameter_(self):
        return self.handle

    def set_stream(self, stream):
        s = stream if isinstance(stream, int) else stream.cuda_stream
        _check(self, _lib.gk_ctx_set_stream(self.handle, P(s)), "gk_ctx_set_stream")

    def close(self):
        if self.handle:
            _lib.gk_ctx_destroy(self.handle)
            self.handle = P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _check(ctx, status, where):
    if status != GK_OK:
        msg = _lib.gk_last_error(ctx.handle).decode() if ctx is not None and ctx.handle else ""
        raise GkError(status, where, msg)
    return status


# ------------------------------------------------------------------ entry points
def gk_set_math(ctx, math):
    return _check(ctx, _lib.gk_set_math(ctx.handle, math), "gk_set_math")


def gk_sync(ctx):
    return _check(ctx, _lib.gk_sync(ctx.handle), "gk_sync")


def gk_launch_count(ctx):
    return _lib.gk_launch_count(ctx.handle)


def gk_selftest_wait_timeout(ctx, limit_ns, arrive, elapsed_ns=None):
    return _check(ctx, _lib.gk_selftest_wait_timeout(ctx.handle, int(limit_ns), int(arrive), _p(elapsed_ns)),
                  "gk_selftest_wait_timeout")


def gk_embedding_fwd(ctx, ids, wte, wpe, x, B, T, C, V):
    return _check(ctx, _lib.gk_embedding_fwd(ctx.handle, _p(ids), _p(wte), _p(wpe), _p(x), B, T, C, V),
                  "gk_embedding_fwd")


def gk_embedding_bwd(ctx, ids, dx, dwte, dwpe, B, T, C, V):
    return _check(ctx, _lib.gk_embedding_bwd(ctx.handle, _p(ids), _p(dx), _p(dwte), _p(dwpe), B, T, C, V),
                  "gk_embedding_bwd")


def gk_layernorm_fwd(ctx, x, gamma, beta, y, y_dtype, mean, rstd, rows, C, eps=1e-5, x_copy=None):
    return _check(ctx, _lib.gk_layernorm_fwd(ctx.handle, _p(x), _p(gamma), _p(beta), _p(y), y_dtype, _p(mean),
                                             _p(rstd), rows, C, eps, _p(x_copy)), "gk_layernorm_fwd")


def gk_layernorm_bwd(ctx, x, gamma, mean, rstd, dy, dx, accumulate_dx, dx_bf16, dgamma, dbeta, rows, C,
                     dx_colsum=None):
    return _check(ctx, _lib.gk_layernorm_bwd(ctx.handle, _p(x), _p(gamma), _p(mean), _p(rstd), _p(dy), _p(dx),
                                             int(accumulate_dx), _p(dx_bf16), _p(dgamma), _p(dbeta), _p(dx_colsum),
                                             rows, C), "gk_layernorm_bwd")


def gk_layernorm_bwd_noalloc(stream, x, gamma, mean, rstd, dy, dx, accumulate_dx, dx_bf16, dgamma, dbeta, rows, C):
    """gk_layernorm_bwd with its scratch in the library's fixed array; `stream` is a cudaStream_t
    (int) or a torch.cuda.Stream. Returns the status code (GkError on failure)."""
    s = stream if isinstance(stream, int) else stream.cuda_stream
    return _check(None, _lib.gk_layernorm_bwd_noalloc(P(s), _p(x), _p(gamma), _p(mean), _p(rstd), _p(dy), _p(dx),
                                                      int(accumulate_dx), _p(dx_bf16), _p(dgamma), _p(dbeta),
                                                      rows, C), "gk_layernorm_bwd_noalloc")


def gk_gelu_fwd(ctx, x, y, n):
    return _check(ctx, _lib.gk_gelu_fwd(ctx.handle, _p(x), _p(y), n), "gk_gelu_fwd")


def gk_gelu_bwd(ctx, x, dy, dx, n):
    return _check(ctx, _lib.gk_gelu_bwd(ctx.handle, _p(x), _p(dy), _p(dx), n), "gk_gelu_bwd")


def gk_matmul_fwd(ctx, dtype, X, ldx, W, ldw, transW, bias, residual, ldr, Y, ldy, y_dtype, N, K, M,
                  act=GK_ACT_NONE, preact=None, ldp=0, X_lo=None, W_lo=None):
    return _check(ctx, _lib.gk_matmul_fwd(ctx.handle, dtype, _p(X), ldx, _p(W), ldw, int(transW), _p(bias),
                                          _p(residual), ldr, _p(Y), ldy, y_dtype, N, K, M, act, _p(preact), ldp,
                                          _p(X_lo), _p(W_lo)), "gk_matmul_fwd")


def gk_matmul_bwd(ctx, dtype, X, ldx, W, ldw, transW, dY, lddy, dX, lddx, dx_dtype, accumulate_dX, preact_X, ldp,
                  dW, lddw, dbias, N, K, M):
    return _check(ctx, _lib.gk_matmul_bwd(ctx.handle, dtype, _p(X), ldx, _p(W), ldw, int(transW), _p(dY), lddy,
                                          _p(dX), lddx, dx_dtype, int(accumulate_dX), _p(preact_X), ldp, _p(dW),
                                          lddw, _p(dbias), N, K, M), "gk_matmul_bwd")


def gk_attn_fwd(ctx, dtype, qkv, y, lse, B, T, H, hs):
    return _check(ctx, _lib.gk_attn_fwd(ctx.handle, dtype, _p(qkv), _p(y), _p(lse), B, T, H, hs), "gk_attn_fwd")


def gk_attn_bwd(ctx, dtype, qkv, y, lse, dy, dqkv, B, T, H, hs):
    return _check(ctx, _lib.gk_attn_bwd(ctx.handle, dtype, _p(qkv), _p(y), _p(lse), _p(dy), _p(dqkv), B, T, H, hs),
                  "gk_attn_bwd")


def gk_softmax_ce_fwd(ctx, logits, ldl, targets, loss, lse, rows, V):
    return _check(ctx, _lib.gk_softmax_ce_fwd(ctx.handle, _p(logits), ldl, _p(targets), _p(loss), _p(lse), rows, V),
                  "gk_softmax_ce_fwd")


def gk_softmax_ce_bwd(ctx, logits, ldl, targets, lse, dloss, dlogits, lddl, dl_dtype, rows, V):
    return _check(ctx, _lib.gk_softmax_ce_bwd(ctx.handle, _p(logits), ldl, _p(targets), _p(lse), _p(dloss),
                                              _p(dlogits), lddl, dl_dtype, rows, V), "gk_softmax_ce_bwd")


def gk_lmhead_ce_fwd(ctx, dtype, X, ldx, W, ldw, targets, loss, lse, N, C, V):
    return _check(ctx, _lib.gk_lmhead_ce_fwd(ctx.handle, dtype, _p(X), ldx, _p(W), ldw, _p(targets), _p(loss), _p(lse),
                                             N, C, V), "gk_lmhead_ce_fwd")


def gk_lmhead_ce_bwd(ctx, dtype, X, ldx, W, ldw, targets, lse, dloss, dX, lddx, accumulate_dX, dW, lddw, scratch,
                     scratch_elems, N, C, V):
    return _check(ctx, _lib.gk_lmhead_ce_bwd(ctx.handle, dtype, _p(X), ldx, _p(W), ldw, _p(targets), _p(lse),
                                             _p(dloss), _p(dX), lddx, int(accumulate_dX), _p(dW), lddw, _p(scratch),
                                             scratch_elems, N, C, V), "gk_lmhead_ce_bwd")


def gk_to_bf16(ctx, x, y, n, y_lo=None):
    return _check(ctx, _lib.gk_to_bf16(ctx.handle, _p(x), _p(y), _p(y_lo), n), "gk_to_bf16")


def gk_adamw_step(ctx, params, lr, beta1, beta2, eps, wd, step, zero_grad=False):
    """params: a list of dicts with keys p, g, m, v, n, decay, p_bf16 (tensors or addresses)."""
    arr = (gk_param * len(params))()
    for i, q in enumerate(params):
        arr[i] = gk_param(_p(q["p"]), _p(q["g"]), _p(q["m"]), _p(q["v"]), int(q["n"]), int(q.get("decay", 0)),
                          _p(q.get("p_bf16")), _p(q.get("p_bf16_lo")))
    return _check(ctx, _lib.gk_adamw_step(ctx.handle, arr, len(params), lr, beta1, beta2, eps, wd, step,
                                          int(zero_grad)), "gk_adamw_step")


def _cfg(V, T, C, H, L):
    return gk_gpt_cfg(V, T, C, H, L)


def gk_gpt_offset(cfg, which, layer=0):
    return _lib.gk_gpt_offset(ct.byref(cfg), which, layer)


def gk_gpt_numel(cfg):
    return _lib.gk_gpt_numel(ct.byref(cfg))


def gk_gpt_n_decay(cfg):
    return _lib.gk_gpt_n_decay(ct.byref(cfg))


class KvCache:
    """A libgk KV cache (gk_kv_create / gk_kv_destroy)."""

    def __init__(self, ctx, cfg, B, Tmax):
        h = P()
        _check(ctx, _lib.gk_kv_create(ctx.handle, ct.byref(h), ct.byref(cfg), B, Tmax), "gk_kv_create")
        self.handle, self.ctx = h, ctx

    def data_ptr(self):
        return _lib.gk_kv_data(self.handle)

    def length(self):
        return _lib.gk_kv_length(self.handle)

    def close(self):
        if self.handle:
            _lib.gk_kv_destroy(self.handle)
            self.handle = P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _sample(s):
    if s is None:
        return None
    top_k, temperature, seed, counter = s
    return ct.byref(gk_sample_cfg(top_k, temperature, seed, counter))


def gk_prefill(ctx, params, kv, ids, Tp, last_logits):
    return _check(ctx, _lib.gk_prefill(ctx.handle, _p(params), kv.handle, _p(ids), Tp, _p(last_logits)),
                  "gk_prefill")


def gk_decode_step(ctx, params, kv, tokens, logits, next_ids, sample=None):
    """sample: None (greedy) or (top_k, temperature, seed, counter)."""
    return _check(ctx, _lib.gk_decode_step(ctx.handle, _p(params), kv.handle, _p(tokens), _p(logits), _p(next_ids),
                                           _sample(sample)), "gk_decode_step")


def gk_decode_run(ctx, params, kv, tokens, logits, next_ids, n_steps, sample=None):
    """n_steps decode steps, each feeding its selection back through tokens (one captured step
    replayed as a CUDA graph). sample: None (greedy) or (top_k, temperature, seed, counter)."""
    return _check(ctx, _lib.gk_decode_run(ctx.handle, _p(params), kv.handle, _p(tokens), _p(logits), _p(next_ids),
                                          _sample(sample), n_steps), "gk_decode_run")


def gk_generate_uncached(ctx, params, kv, ids, Tp, n_new, logits, sample=None):
    """n_new tokens by re-running the whole prefix per token: ids [B, Tp + n_new] (device int32)
    holds the prompt in its first Tp columns and receives the selections."""
    return _check(ctx, _lib.gk_generate_uncached(ctx.handle, _p(params), kv.handle, _p(ids), Tp, n_new, _p(logits),
                                                 _sample(sample)), "gk_generate_uncached")


# ---- generic ops of the autograd engine (float32 device tensors of n elements) and SGD
def gk_add_fwd(ctx, a, b, y, n, m):
    return _check(ctx, _lib.gk_add_fwd(ctx.handle, _p(a), _p(b), _p(y), n, m), "gk_add_fwd")


def gk_add_bwd(ctx, g, da, db, n, m, accumulate=0):
    return _check(ctx, _lib.gk_add_bwd(ctx.handle, _p(g), _p(da), _p(db), n, m, accumulate), "gk_add_bwd")


def gk_mul_fwd(ctx, a, b, y, n):
    return _check(ctx, _lib.gk_mul_fwd(ctx.handle, _p(a), _p(b), _p(y), n), "gk_mul_fwd")


def gk_mul_bwd(ctx, g, a, b, da, db, n, accumulate=0):
    return _check(ctx, _lib.gk_mul_bwd(ctx.handle, _p(g), _p(a), _p(b), _p(da), _p(db), n, accumulate),
                  "gk_mul_bwd")


def gk_scale_fwd(ctx, a, s, y, n):
    return _check(ctx, _lib.gk_scale_fwd(ctx.handle, _p(a), s, _p(y), n), "gk_scale_fwd")


def gk_scale_bwd(ctx, g, s, da, n, accumulate=0):
    return _check(ctx, _lib.gk_scale_bwd(ctx.handle, _p(g), s, _p(da), n, accumulate), "gk_scale_bwd")


def gk_sum_fwd(ctx, a, y, n):
    return _check(ctx, _lib.gk_sum_fwd(ctx.handle, _p(a), _p(y), n), "gk_sum_fwd")


def gk_sum_bwd(ctx, g, da, n, accumulate=0):
    return _check(ctx, _lib.gk_sum_bwd(ctx.handle, _p(g), _p(da), n, accumulate), "gk_sum_bwd")


def gk_tanh_fwd(ctx, x, y, n):
    return _check(ctx, _lib.gk_tanh_fwd(ctx.handle, _p(x), _p(y), n), "gk_tanh_fwd")


def gk_tanh_bwd(ctx, y, g, dx, n, accumulate=0):
    return _check(ctx, _lib.gk_tanh_bwd(ctx.handle, _p(y), _p(g), _p(dx), n, accumulate), "gk_tanh_bwd")


def gk_sgd_step(ctx, p, g, n, lr):
    return _check(ctx, _lib.gk_sgd_step(ctx.handle, _p(p), _p(g), n, lr), "gk_sgd_step")


def gk_sample(ctx, kv, logits, ld, next_ids, sample=None):
    return _check(ctx, _lib.gk_sample(ctx.handle, kv.handle, _p(logits), ld, _p(next_ids), _sample(sample)),
                  "gk_sample")


# ---- safetensors files of float32 tensors (host code in libgk; arrays on the host or the GPU)
def _st_check(status, where):
    if status != GK_OK:
        raise GkError(status, where, _lib.gk_st_last_error().decode())


class SafeTensors:
    """An open safetensors file: names (header order), shapes, dtypes, metadata, and reads of
    float32 tensors into new host arrays or into given host / CUDA tensors."""

    def __init__(self, path):
        h = P()
        _st_check(_lib.gk_st_open(os.fsencode(path), ct.byref(h)), "gk_st_open")
        self.handle = h

    def close(self):
        if self.handle:
            _lib.gk_st_close(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def names(self):
        return [_lib.gk_st_name(self.handle, i).decode() for i in range(_lib.gk_st_count(self.handle))]

    def _index(self, name):
        i = _lib.gk_st_find(self.handle, name.encode())
        if i < 0:
            raise KeyError(name)
        return i

    def shape(self, name):
        i = self._index(name)
        sh = _lib.gk_st_shape(self.handle, i)
        return tuple(sh[k] for k in range(_lib.gk_st_ndim(self.handle, i)))

    def dtype(self, name):
        return _lib.gk_st_dtype(self.handle, self._index(name)).decode()

    def metadata(self, key):
        v = _lib.gk_st_metadata(self.handle, key.encode())
        return None if v is None else v.decode()

    def read(self, name, out=None):
        """Into `out` (a contiguous float32 torch tensor, host or CUDA) or a new numpy array."""
        import numpy as np

        i = self._index(name)
        if out is None:
            arr = np.empty(self.shape(name), np.float32)
            _st_check(_lib.gk_st_read_f32(self.handle, i, arr.ctypes.data, arr.size, 0), "gk_st_read_f32")
            return arr
        _st_check(_lib.gk_st_read_f32(self.handle, i, out.data_ptr(), out.numel(), int(out.is_cuda)),
                  "gk_st_read_f32")
        return out


def write_safetensors(path, tensors, metadata=None):
    """tensors: (name, array) pairs or a dict, each a float32 numpy array or a contiguous
    float32 torch tensor (all on the host, or all on the GPU); metadata: str -> str."""
    import numpy as np

    items = list(tensors.items()) if isinstance(tensors, dict) else list(tensors)
    keep, ptrs, ndims, shapes = [], [], [], []
    on_dev = 0
    for _, a in items:
        if hasattr(a, "data_ptr"):
            on_dev = int(a.is_cuda)
            keep.append(a)
            ptrs.append(a.data_ptr())
        else:
            a = np.require(a, dtype=np.float32, requirements="C")  # keeps 0-d arrays 0-d
            keep.append(a)
            ptrs.append(a.ctypes.data)
        ndims.append(len(a.shape))
        shapes += list(a.shape)
    n, meta = len(items), list((metadata or {}).items())
    names = (ct.c_char_p * max(n, 1))(*[k.encode() for k, _ in items])
    mk = (ct.c_char_p * max(len(meta), 1))(*[str(k).encode() for k, _ in meta])
    mv = (ct.c_char_p * max(len(meta), 1))(*[str(v).encode() for _, v in meta])
    _st_check(_lib.gk_st_write_f32(os.fsencode(path), n, names, (I32 * max(n, 1))(*ndims),
                                   (I64 * max(len(shapes), 1))(*shapes), (P * max(n, 1))(*ptrs), on_dev, len(meta),
                                   mk, mv), "gk_st_write_f32")
