"""Single-op parity of libgk's CUDA kernels against the oracle, through the C ABI.

Sizes cover the op sweep (MatMul/MatMulT at 256, 1024, 4096 and 4096x768x3072; LayerNorm,
GELU and softmax-CE on [4096, 768] and [4096, 50257]) plus ragged shapes that leave partial
tiles, and the degenerate cases. Tolerances: float32 kernels are compared with the float64
oracle on the same float32 inputs; bf16-operand kernels with the oracle on the same
bf16-rounded operands, so both measure the kernel's own accumulation error only.
"""
import numpy as np
import pytest

import synth
from oracle import ops
from tests.conftest import assert_close, rel_l2

pytestmark = pytest.mark.gpu


def _t():
    import torch

    return torch


def dev(a, dtype=None):
    torch = _t()
    t = torch.as_tensor(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    return t.float().cpu().numpy() if t.dtype != _t().int32 else t.cpu().numpy()


def bf16_round(a):
    torch = _t()
    return torch.as_tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def normal(seed, *shape, std=1.0):
    return synth.Stream(seed).normal(int(np.prod(shape)), std).reshape(shape)


# ----------------------------------------------------------------------- embedding
@pytest.mark.parametrize("B,T,C,V", [(2, 5, 12, 9), (4, 1024, 768, 50257), (3, 7, 96, 3)])
def test_embedding_fwd_exact(gkctx, B, T, C, V):
    from gpt_decoder_gb300 import gk

    st = synth.Stream(100 + C)
    ids = st.ints(B * T, V).reshape(B, T)
    wte, wpe = st.normal(V * C).reshape(V, C), st.normal(T * C).reshape(T, C)
    x = _t().empty(B * T, C, device="cuda")
    gk.gk_embedding_fwd(gkctx, dev(ids.reshape(-1)), dev(wte), dev(wpe), x, B, T, C, V)
    gk.gk_sync(gkctx)
    ref = ops.embedding_fwd(ids, wte, wpe).reshape(B * T, C).astype(np.float32)
    assert np.array_equal(host(x), ref)


def test_embedding_bad_id_reports_index_error(gkctx):
    from gpt_decoder_gb300 import gk

    x = _t().empty(2, 4, device="cuda")
    ids = dev(np.array([1, 9], dtype=np.int32))
    gk.gk_embedding_fwd(gkctx, ids, dev(np.ones((5, 4), np.float32)), dev(np.ones((2, 4), np.float32)), x, 1, 2, 4, 5)
    with pytest.raises(gk.GkError) as e:
        gk.gk_sync(gkctx)
    assert e.value.status == gk.GK_ERR_INDEX
    gk.gk_sync(gkctx)  # the error word was cleared
    assert np.array_equal(host(x)[1], np.zeros(4, np.float32))


@pytest.mark.parametrize("B,T,C,V", [(3, 4, 6, 5), (8, 64, 96, 64), (4, 1024, 768, 50257), (16, 1024, 768, 50257)])
def test_embedding_bwd_bit_exact(gkctx, B, T, C, V):
    from gpt_decoder_gb300 import gk

    st = synth.Stream(200 + B)
    ids = st.ints(B * T, V).reshape(B, T)
    if V > 1000:
        ids[:, ::7] = 17  # many repeats of one token
    dx = st.normal(B * T * C).reshape(B * T, C)
    dwte0 = st.normal(V * C, 0.1).reshape(V, C)
    dwpe0 = st.normal(T * C, 0.1).reshape(T, C)
    g_te, g_pe = dev(dwte0), dev(dwpe0)
    gk.gk_embedding_bwd(gkctx, dev(ids.reshape(-1)), dev(dx), g_te, g_pe, B, T, C, V)
    gk.gk_sync(gkctx)
    r_te, r_pe = dwte0.copy(), dwpe0.copy()
    ops.embedding_bwd(ids, dx, r_te, r_pe)
    assert np.array_equal(host(g_te), r_te)
    assert np.array_equal(host(g_pe), r_pe)


# ----------------------------------------------------------------------- layernorm
@pytest.mark.parametrize("rows,C", [(4096, 768), (4096, 50257), (37, 96), (5, 130), (1, 1024), (3, 7), (64, 8192),
                                    (9, 5003)])
@pytest.mark.parametrize("ydt", ["f32", "bf16"])
def test_layernorm_fwd(gkctx, rows, C, ydt):
    from gpt_decoder_gb300 import gk

    if C == 50257 and ydt == "bf16":
        pytest.skip("covered in float32")
    x = normal(300 + C, rows, C) * 2 + 0.5
    gm, bt = normal(301, C), normal(302, C)
    torch = _t()
    y = torch.empty(rows, C, device="cuda", dtype=torch.float32 if ydt == "f32" else torch.bfloat16)
    mean, rstd = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
    xc = torch.full((rows, C), float("nan"), device="cuda")
    gk.gk_layernorm_fwd(gkctx, dev(x), dev(gm), dev(bt), y, gk.GK_F32 if ydt == "f32" else gk.GK_BF16, mean, rstd,
                        rows, C, 1e-5, x_copy=xc)
    gk.gk_sync(gkctx)
    assert np.array_equal(host(xc), x.astype(np.float32))  # the residual-stream copy is exact
    ry, rm, rr = ops.layernorm_fwd(x, gm, bt)
    tol = 2e-5 if ydt == "f32" else 2e-2
    assert np.abs(host(y) - ry).max() < tol * max(1.0, np.abs(ry).max() / 4)
    np.testing.assert_allclose(host(mean), rm, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(host(rstd), rr, rtol=2e-5)


@pytest.mark.parametrize("rows,C", [(4096, 768), (4096, 50257), (37, 96), (5, 130), (1, 1024)])
@pytest.mark.parametrize("acc", [0, 1])
def test_layernorm_bwd(gkctx, rows, C, acc):
    from gpt_decoder_gb300 import gk

    torch = _t()
    x = normal(310 + C, rows, C) * 2 + 0.5
    gm, bt = normal(311, C), normal(312, C)
    g = normal(313, rows, C)
    _, rm, rr = ops.layernorm_fwd(x, gm, bt)
    dx0 = normal(314, rows, C)
    dg0, db0 = normal(315, C), normal(316, C)
    ds0 = normal(317, C)
    dx, dgm, dbt, dsum = dev(dx0), dev(dg0), dev(db0), dev(ds0)
    dxb = torch.empty(rows, C, device="cuda", dtype=torch.bfloat16)
    gk.gk_layernorm_bwd(gkctx, dev(x), dev(gm), dev(rm.astype(np.float32)), dev(rr.astype(np.float32)), dev(g), dx,
                        acc, dxb, dgm, dbt, rows, C, dx_colsum=dsum)
    gk.gk_sync(gkctx)
    rdx, rdg, rdb = ops.layernorm_bwd(x, gm, rm.astype(np.float32), rr.astype(np.float32), g)
    if acc:
        rdx = rdx + dx0
    assert_close(host(dx), rdx, 1e-5)
    assert_close(host(dxb), host(dx), 5e-3)
    assert_close(host(dgm), rdg + dg0, 1e-5)
    assert_close(host(dbt), rdb + db0, 1e-5)
    # the column sums of the resulting dx (a bias gradient): the oracle's bias backward of dx
    assert_close(host(dsum), ops.bias_bwd(rdx) + ds0, 1e-5)


# ---------------------------------------------------------------------------- GELU
@pytest.mark.parametrize("n", [4096 * 768, 4096 * 50257, 1, 1023])
def test_gelu(gkctx, n):
    from gpt_decoder_gb300 import gk

    torch = _t()
    x = normal(400, n) * 3
    g = normal(401, n)
    y, dx = torch.empty(n, device="cuda"), torch.empty(n, device="cuda")
    dxx = dev(x)
    gk.gk_gelu_fwd(gkctx, dxx, y, n)
    gk.gk_gelu_bwd(gkctx, dxx, dev(g), dx, n)
    gk.gk_sync(gkctx)
    assert np.abs(host(y) - ops.gelu_fwd(x)).max() < 1e-5
    assert np.abs(host(dx) - ops.gelu_bwd(x, g)).max() < 2e-5


# -------------------------------------------------------------------------- MatMul
@pytest.fixture(params=["f32", "3xtf32"])
def f32_math(request):
    """The float32 products' arithmetic: "f32" float32 FMA on the CUDA cores, "3xtf32" the
    tensor cores (the context's default)."""
    return request.param


SWEEP = [(256, 256, 256), (1024, 1024, 1024), (4096, 4096, 4096), (4096, 768, 3072)]
RAGGED = [(131, 67, 45), (1, 5, 3), (200, 1, 130), (129, 129, 257)]


def _set_math(gkctx, dt):
    """dt "f32": float32 operands, float32 FMA; "3xtf32": float32 operands on the tensor cores;
    "bf16": bf16 operands. Returns the operand type ("f32" or "bf16")."""
    from gpt_decoder_gb300 import gk

    gk.gk_set_math(gkctx, gk.GK_MATH_FP32 if dt == "f32" else gk.GK_MATH_3XTF32)
    return "f32" if dt == "3xtf32" else dt


def _tol(dt, K, base=2e-5):
    """Element-wise tolerance (relative to max|ref|) of a product with reduction length K.
    3xTF32: the three TF32 products are exact, but every tcgen05 MMA (K = 8) adds into the
    float32 accumulator in tensor memory with truncation, so up to 3 * ceil(K / 8) one-ulp
    losses of the running sum add up in one direction (measured: 3.4e-5 of max|y| at K = 4096,
    against 7e-7 for the FMA kernel)."""
    return max(base, 3 * -(-K // 8) * 2.0 ** -24) if dt == "3xtf32" else base


def _restore_math(gkctx):
    from gpt_decoder_gb300 import gk

    gk.gk_set_math(gkctx, gk.GK_MATH_3XTF32)


def _matmul_case(gkctx, N, K, M, transW, dt, bias, resid, act, seed):
    from gpt_decoder_gb300 import gk

    torch = _t()
    dt = _set_math(gkctx, dt)
    x = normal(seed, N, K)
    w = normal(seed + 1, M, K) if transW else normal(seed + 1, K, M)
    if dt == "bf16":
        x, w = bf16_round(x), bf16_round(w)
    b = normal(seed + 2, M) if bias else None
    r = normal(seed + 3, N, M) if resid else None
    gdt = gk.GK_F32 if dt == "f32" else gk.GK_BF16
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    y = torch.empty(N, M, device="cuda")
    pre = torch.empty(N, M, device="cuda") if act else None
    gk.gk_matmul_fwd(gkctx, gdt, dev(x, tdt), K, dev(w, tdt), w.shape[1], transW, None if b is None else dev(b),
                     None if r is None else dev(r), M, y, M, gk.GK_F32, N, K, M,
                     gk.GK_ACT_GELU if act else gk.GK_ACT_NONE, pre, M)
    gk.gk_sync(gkctx)
    _restore_math(gkctx)
    ref = ops.matmul_t_fwd(x, w) if transW else ops.matmul_fwd(x, w)
    if b is not None:
        ref = ref + b
    if r is not None:
        ref = ref + r
    if act:
        assert_close(host(pre), ref, 2e-5)
        ref = ops.gelu_fwd(ref)
    return host(y), ref


@pytest.mark.parametrize("N,K,M", SWEEP + RAGGED)
@pytest.mark.parametrize("transW", [0, 1])
def test_matmul_fwd_f32(gkctx, f32_math, N, K, M, transW):
    y, ref = _matmul_case(gkctx, N, K, M, transW, f32_math, True, False, False, 500)
    assert_close(y, ref, _tol(f32_math, K))


@pytest.mark.parametrize("N,K,M", [(4096, 768, 3072), (512, 96, 288), (131, 67, 45), (256, 256, 256),
                                   (1160, 200, 520), (640, 64, 256)])
@pytest.mark.parametrize("transW", [0, 1])
def test_matmul_fwd_bf16_operands(gkctx, N, K, M, transW):
    y, ref = _matmul_case(gkctx, N, K, M, transW, "bf16", True, False, False, 510)
    assert_close(y, ref, 2e-5)


@pytest.mark.parametrize("dt", ["f32", "3xtf32", "bf16"])
def test_matmul_fwd_epilogues(gkctx, dt):
    y, ref = _matmul_case(gkctx, 300, 96, 384, 0, dt, True, True, False, 520)
    assert_close(y, ref, 2e-5)
    y, ref = _matmul_case(gkctx, 300, 96, 384, 0, dt, True, False, True, 530)
    assert_close(y, ref, 2e-5)


@pytest.mark.parametrize("dt", ["f32", "3xtf32", "bf16"])
@pytest.mark.parametrize("N,K,M", [(300, 96, 384), (4096, 768, 768), (77, 64, 200)])
def test_matmul_in_place_residual_is_bit_identical(gkctx, dt, N, K, M):
    """Y = X W + b + Y in place (an accumulation, TMA reduce-add on the tensor cores) equals
    the out-of-place residual result bit for bit."""
    from gpt_decoder_gb300 import gk

    torch = _t()
    dt = _set_math(gkctx, dt)
    x, w, b, r = normal(540, N, K), normal(541, K, M), normal(542, M), normal(543, N, M)
    if dt == "bf16":
        x, w = bf16_round(x), bf16_round(w)
    gdt = gk.GK_F32 if dt == "f32" else gk.GK_BF16
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    dx_, dw_, db_ = dev(x, tdt), dev(w, tdt), dev(b)
    y_out = torch.empty(N, M, device="cuda")
    gk.gk_matmul_fwd(gkctx, gdt, dx_, K, dw_, M, 0, db_, dev(r), M, y_out, M, gk.GK_F32, N, K, M)
    y_in = dev(r)
    gk.gk_matmul_fwd(gkctx, gdt, dx_, K, dw_, M, 0, db_, y_in, M, y_in, M, gk.GK_F32, N, K, M)
    gk.gk_sync(gkctx)
    _restore_math(gkctx)
    assert np.array_equal(host(y_in), host(y_out))
    assert_close(host(y_in), ops.matmul_fwd(x, w) + b + r, 2e-5)


@pytest.mark.parametrize("N,K,M,act", [(1000, 3000, 1500, False), (1000, 700, 1500, True), (37, 5000, 300, False)])
def test_matmul_3xtf32_in_chunks(N, K, M, act):
    """3xTF32 products whose TF32 planes do not fit the context's workspace (4 MiB here) run in
    blocks of rows and columns, and (plain sums) in K slices added into Y; the result, bias,
    GELU epilogue and the backward's dX and dW included, matches the oracle."""
    import torch

    from gpt_decoder_gb300 import gk

    ctx = gk.Ctx(torch.cuda.current_stream().cuda_stream, workspace_bytes=4 << 20)
    try:
        gk.gk_set_math(ctx, gk.GK_MATH_3XTF32)
        x, w, b = normal(700, N, K), normal(701, K, M), normal(702, M)
        y = torch.empty(N, M, device="cuda")
        pre = torch.empty(N, M, device="cuda") if act else None
        gk.gk_matmul_fwd(ctx, gk.GK_F32, dev(x), K, dev(w), M, 0, dev(b), None, 0, y, M, gk.GK_F32, N, K, M,
                         gk.GK_ACT_GELU if act else gk.GK_ACT_NONE, pre, M)
        g = normal(703, N, M)
        dx, dw = torch.empty(N, K, device="cuda"), torch.zeros(K, M, device="cuda")
        gk.gk_matmul_bwd(ctx, gk.GK_F32, dev(x), K, dev(w), M, 0, dev(g), M, dx, K, gk.GK_F32, 0, None, 0, dw, M,
                         None, N, K, M)
        gk.gk_sync(ctx)
    finally:
        ctx.close()
    ref = ops.matmul_fwd(x, w) + b
    if act:
        assert_close(host(pre), ref, _tol("3xtf32", K), "preact")
        ref = ops.gelu_fwd(ref)
    assert_close(host(y), ref, _tol("3xtf32", K), "y")
    rdx, rdw = ops.matmul_bwd(x, w, g)
    assert_close(host(dx), rdx, _tol("3xtf32", M), "dx")
    assert_close(host(dw), rdw, _tol("3xtf32", N), "dw")


def _matmul_bwd_case(gkctx, N, K, M, transW, dt, acc, gelu, seed):
    from gpt_decoder_gb300 import gk

    torch = _t()
    dt = _set_math(gkctx, dt)
    x = normal(seed, N, K)
    w = normal(seed + 1, M, K) if transW else normal(seed + 1, K, M)
    g = normal(seed + 2, N, M)
    pre = normal(seed + 3, N, K) if gelu else None
    if dt == "bf16":
        x, w, g = bf16_round(x), bf16_round(w), bf16_round(g)
        if gelu:
            pre = bf16_round(pre)
    gdt = gk.GK_F32 if dt == "f32" else gk.GK_BF16
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    dx0 = normal(seed + 4, N, K)
    dw0 = normal(seed + 5, *w.shape)
    db0 = normal(seed + 6, M)
    dx, dw, db = dev(dx0), dev(dw0), dev(db0)
    gk.gk_matmul_bwd(gkctx, gdt, dev(x, tdt), K, dev(w, tdt), w.shape[1], transW, dev(g, tdt), M, dx, K, gk.GK_F32,
                     acc, None if pre is None else dev(pre, tdt), K, dw, w.shape[1], db, N, K, M)
    gk.gk_sync(gkctx)
    _restore_math(gkctx)
    rdx, rdw = (ops.matmul_t_bwd(x, w, g) if transW else ops.matmul_bwd(x, w, g))
    if gelu:
        rdx = ops.gelu_bwd(pre, rdx)
    if acc:
        rdx = rdx + dx0
    return (host(dx), rdx), (host(dw), rdw + dw0), (host(db), ops.bias_bwd(g) + db0)


@pytest.mark.parametrize("N,K,M", SWEEP + RAGGED)
@pytest.mark.parametrize("transW", [0, 1])
def test_matmul_bwd_f32(gkctx, f32_math, N, K, M, transW):
    (dx, rdx), (dw, rdw), (db, rdb) = _matmul_bwd_case(gkctx, N, K, M, transW, f32_math, 0, False, 600)
    assert_close(dx, rdx, _tol(f32_math, M))
    assert_close(dw, rdw, _tol(f32_math, N))
    assert_close(db, rdb, 2e-5)


@pytest.mark.parametrize("N,K,M", [(4096, 768, 3072), (512, 96, 288), (131, 67, 45), (1160, 520, 200)])
@pytest.mark.parametrize("transW", [0, 1])
def test_matmul_bwd_bf16_operands(gkctx, N, K, M, transW):
    (dx, rdx), (dw, rdw), (db, rdb) = _matmul_bwd_case(gkctx, N, K, M, transW, "bf16", 1, False, 610)
    assert_close(dx, rdx, 2e-5)
    assert_close(dw, rdw, 2e-5)
    assert_close(db, rdb, 2e-5)


@pytest.mark.parametrize("dt", ["f32", "3xtf32", "bf16"])
def test_matmul_bwd_fused_gelu(gkctx, dt):
    (dx, rdx), _, _ = _matmul_bwd_case(gkctx, 300, 384, 96, 0, dt, 0, True, 620)
    assert_close(dx, rdx, (5e-3 if dt == "bf16" else 2e-5))


@pytest.mark.parametrize("dt", ["f32", "3xtf32", "bf16"])
def test_matmul_bwd_fused_gelu_accumulates_after_the_gelu_factor(gkctx, dt):
    """accumulate_dX with preact_X: dX_old + (dY W^T) * gelu'(preact)."""
    (dx, rdx), (dw, rdw), _ = _matmul_bwd_case(gkctx, 300, 384, 96, 0, dt, 1, True, 625)
    assert_close(dx, rdx, (5e-3 if dt == "bf16" else 2e-5))
    assert_close(dw, rdw, 2e-5)


# bf16 results through the tensor-core epilogue: ragged rows and columns (partial 32-row
# groups, partial chunks, idle column halves) next to full tiles
# (with at least four 128-row tiles the products run on CTA pairs: an odd tile count leaves the
# last pair's second CTA past the rows, 700 leaves it a partial tile)
BF16_OUT = [(4096, 768, 3072), (300, 96, 384), (131, 64, 45), (77, 128, 200), (1, 64, 8), (333, 96, 130),
            (257, 64, 520), (640, 96, 384), (700, 200, 520)]


@pytest.mark.parametrize("N,K,M", BF16_OUT)
@pytest.mark.parametrize("mode", ["plain", "gelu", "dgelu"])
def test_matmul_bf16_results(gkctx, N, K, M, mode):
    from gpt_decoder_gb300 import gk

    torch = _t()
    seed = 640 + N + M
    x, w, b = bf16_round(normal(seed, N, K)), bf16_round(normal(seed + 1, K, M)), normal(seed + 2, M)
    bf = torch.bfloat16
    if mode == "dgelu":
        # dX [N, K] = (dY [N, M] W^T) * gelu'(pre), all bf16
        g, pre = bf16_round(normal(seed + 3, N, M)), bf16_round(normal(seed + 4, N, K))
        dx = torch.full((N, K), float("nan"), dtype=bf, device="cuda")
        gk.gk_matmul_bwd(gkctx, gk.GK_BF16, None, 0, dev(w, bf), M, 0, dev(g, bf), M, dx, K, gk.GK_BF16, 0,
                         dev(pre, bf), K, None, 0, None, N, K, M)
        gk.gk_sync(gkctx)
        rdx, _ = ops.matmul_bwd(x, w, g)
        assert_close(dx.float().cpu().numpy(), ops.gelu_bwd(pre, rdx), 5e-3)
        return
    y = torch.full((N, M), float("nan"), dtype=bf, device="cuda")
    pre = torch.full((N, M), float("nan"), dtype=bf, device="cuda") if mode == "gelu" else None
    gk.gk_matmul_fwd(gkctx, gk.GK_BF16, dev(x, bf), K, dev(w, bf), M, 0, dev(b), None, 0, y, M, gk.GK_BF16, N, K, M,
                     gk.GK_ACT_GELU if mode == "gelu" else gk.GK_ACT_NONE, pre, M)
    gk.gk_sync(gkctx)
    ref = ops.matmul_fwd(x, w) + b
    if mode == "gelu":
        assert_close(pre.float().cpu().numpy(), ref, 5e-3)
        ref = ops.gelu_fwd(ref)
    assert_close(y.float().cpu().numpy(), ref, 5e-3)


def test_matmul_rejects_bad_strides(gkctx):
    from gpt_decoder_gb300 import gk

    x = _t().zeros(4, 4, device="cuda")
    with pytest.raises(gk.GkError) as e:
        gk.gk_matmul_fwd(gkctx, gk.GK_F32, x, 3, x, 4, 0, None, None, 0, x, 4, gk.GK_F32, 4, 4, 4)
    assert e.value.status == gk.GK_ERR_ARG


# ----------------------------------------------------------------------- attention
ATTN = [(2, 64, 4, 24), (1, 77, 2, 64), (2, 1024, 12, 64), (1, 1, 3, 32), (3, 33, 2, 8)]


def _attn_inputs(B, T, H, hs, seed, dt):
    qkv = normal(seed, B, T, 3 * H * hs)
    dy = normal(seed + 1, B, T, H * hs)
    if dt == "bf16":
        qkv, dy = bf16_round(qkv), bf16_round(dy)
    return qkv, dy


@pytest.mark.parametrize("B,T,H,hs", ATTN + [(1, 256, 3, 32), (2, 384, 2, 64)])
@pytest.mark.parametrize("dt", ["f32", "3xtf32", "bf16"])
def test_attention_fwd_bwd(gkctx, B, T, H, hs, dt):
    """f32: float32 FMA on the CUDA cores; 3xtf32: the products on the tensor cores (T a multiple of
    128, other shapes take the float32 kernels); bf16: the bf16 tensor-core kernels (hs = 64)."""
    _attention_case(gkctx, B, T, H, hs, dt)


@pytest.mark.parametrize("B,T,H,hs", [(4, 1024, 12, 64), (8, 300, 12, 64)])
def test_attention_bf16_several_work_items_per_cta(gkctx, B, T, H, hs):
    """The persistent bf16 kernels with more work items than SMs (forward 192, backward 384 and
    288 items), so CTAs carry barrier phases and buffers from one item to the next; T = 300 also
    has items whose second query tile is missing and a ragged last tile."""
    _attention_case(gkctx, B, T, H, hs, "bf16")


def _attention_case(gkctx, B, T, H, hs, dt):
    from gpt_decoder_gb300 import gk

    torch = _t()
    math_dt = dt
    dt = _set_math(gkctx, dt)
    qkv, dy = _attn_inputs(B, T, H, hs, 700 + T, dt)
    gdt = gk.GK_F32 if dt == "f32" else gk.GK_BF16
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    C = H * hs
    d_qkv = dev(qkv.reshape(B * T, 3 * C), tdt)
    y = torch.empty(B * T, C, device="cuda", dtype=tdt)
    lse = torch.empty(B * H * T, device="cuda")
    gk.gk_attn_fwd(gkctx, gdt, d_qkv, y, lse, B, T, H, hs)
    ry, P, rl = ops.attention_fwd(qkv, H)
    gk.gk_sync(gkctx)
    tol_y = _tol(math_dt, T, 2e-5) if dt == "f32" else 8e-3
    assert_close(host(y), ry.reshape(B * T, C), tol_y)
    np.testing.assert_allclose(host(lse), rl.reshape(-1), rtol=1e-5, atol=1e-5)
    dqkv = torch.empty(B * T, 3 * C, device="cuda", dtype=tdt)
    # backward from the oracle's own y (so the test isolates the backward kernel)
    y_in = dev(ry.reshape(B * T, C), tdt)
    gk.gk_attn_bwd(gkctx, gdt, d_qkv, y_in, dev(rl.reshape(-1).astype(np.float32)), dev(dy.reshape(B * T, C), tdt),
                   dqkv, B, T, H, hs)
    gk.gk_sync(gkctx)
    _restore_math(gkctx)
    rd = ops.attention_bwd(qkv, P, dy, H).reshape(B * T, 3 * C)
    assert_close(host(dqkv), rd, (_tol(math_dt, T, 5e-5) if dt == "f32" else 1e-2))


# --------------------------------------------------------- softmax cross-entropy
@pytest.mark.parametrize("rows,V,ldl", [(4096, 768, 768), (4096, 50257, 50257), (4096, 50257, 50304), (7, 3, 8),
                                        (1, 64, 64)])
@pytest.mark.parametrize("dl_dt", ["f32", "bf16"])
def test_softmax_ce(gkctx, rows, V, ldl, dl_dt):
    from gpt_decoder_gb300 import gk

    torch = _t()
    x = np.zeros((rows, ldl), np.float32)
    x[:, :V] = normal(800 + V, rows, V) * 3
    x[:, V:] = np.nan  # padding is never read
    tg = synth.Stream(801).ints(rows, V)
    loss = torch.zeros(1, device="cuda")
    lse = torch.empty(rows, device="cuda")
    dx = dev(x)
    gk.gk_softmax_ce_fwd(gkctx, dx, ldl, dev(tg), loss, lse, rows, V)
    rloss, rlse = ops.softmax_ce_fwd(x[:, :V], tg)
    gk.gk_sync(gkctx)
    assert abs(loss.item() - rloss) < 1e-5 * max(1.0, abs(rloss))
    np.testing.assert_allclose(host(lse), rlse, rtol=1e-6, atol=1e-5)
    dloss = dev(np.array([0.75], np.float32))
    tdt = torch.float32 if dl_dt == "f32" else torch.bfloat16
    dl = torch.full((rows, ldl), 7.0, device="cuda", dtype=tdt)
    gk.gk_softmax_ce_bwd(gkctx, dx, ldl, dev(tg), dev(rlse.astype(np.float32)), dloss, dl, ldl,
                         gk.GK_F32 if dl_dt == "f32" else gk.GK_BF16, rows, V)
    gk.gk_sync(gkctx)
    rd = ops.softmax_ce_bwd(x[:, :V], tg, rlse.astype(np.float32), 0.75)
    got = host(dl)
    assert_close(got[:, :V], rd, (1e-5 if dl_dt == "f32" else 5e-3))
    assert np.all(got[:, V:] == 0)


# ------------------------------------------------------- fused LM head + cross-entropy
@pytest.mark.parametrize("N,C,V", [(300, 96, 50), (512, 128, 1000), (77, 64, 513), (1024, 768, 50257)])
def test_lmhead_ce_fused(gkctx, N, C, V):
    """Loss, LSE, dX and dW of the fused head against the oracle's MatMulT + SoftmaxCE, with
    the backward both in one vocabulary chunk and in chunks of 256 columns."""
    from gpt_decoder_gb300 import gk

    torch = _t()
    seed = 1300 + V
    x = bf16_round(normal(seed, N, C))
    w = bf16_round(normal(seed + 1, V, C) * 0.5)
    tg = synth.Stream(seed + 2).ints(N, V).astype(np.int32)
    dloss = 1.7
    logits = ops.matmul_t_fwd(x, w)
    rloss, rlse = ops.softmax_ce_fwd(logits, tg)
    rdl = ops.softmax_ce_bwd(logits, tg, rlse, dloss)
    rdx, rdw = ops.matmul_t_bwd(x, w, rdl)
    bf = torch.bfloat16
    dx_, w_, t_ = dev(x, bf), dev(w, bf), dev(tg)
    loss = torch.empty(1, device="cuda")
    lse = torch.empty(N, device="cuda")
    gk.gk_lmhead_ce_fwd(gkctx, gk.GK_BF16, dx_, C, w_, C, t_, loss, lse, N, C, V)
    gk.gk_sync(gkctx)
    assert abs(loss.item() - rloss) < 1e-4 * max(1.0, abs(rloss))
    assert np.abs(host(lse) - rlse).max() < 1e-4 * max(1.0, np.abs(rlse).max())
    dl = dev(np.array([dloss], dtype=np.float32))
    dx0, dw0 = normal(seed + 3, N, C), normal(seed + 4, V, C)
    for scratch_cols in (V + 300, 256):
        dx, dw = dev(dx0), dev(dw0)
        scratch = torch.empty(N * scratch_cols, dtype=bf, device="cuda")
        gk.gk_lmhead_ce_bwd(gkctx, gk.GK_BF16, dx_, C, w_, C, t_, lse, dl, dx, C, 1, dw, C, scratch, N * scratch_cols,
                            N, C, V)
        gk.gk_sync(gkctx)
        # dlogits pass through bf16 once: about 2^-9 relative
        assert_close(host(dx) - dx0, rdx, 5e-3, scratch_cols)
        assert_close(host(dw) - dw0, rdw, 5e-3, scratch_cols)


def test_lmhead_ce_reports_bad_target_and_small_scratch(gkctx):
    from gpt_decoder_gb300 import gk

    torch = _t()
    N, C, V = 64, 64, 300
    x = dev(bf16_round(normal(1400, N, C)), torch.bfloat16)
    w = dev(bf16_round(normal(1401, V, C)), torch.bfloat16)
    tg = np.zeros(N, dtype=np.int32)
    tg[5] = V
    loss, lse = torch.empty(1, device="cuda"), torch.empty(N, device="cuda")
    gk.gk_lmhead_ce_fwd(gkctx, gk.GK_BF16, x, C, w, C, dev(tg), loss, lse, N, C, V)
    with pytest.raises(gk.GkError) as e:
        gk.gk_sync(gkctx)
    assert e.value.status == gk.GK_ERR_INDEX
    scratch = torch.empty(N * 255, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gk.GkError) as e:
        gk.gk_lmhead_ce_bwd(gkctx, gk.GK_BF16, x, C, w, C, dev(np.zeros(N, np.int32)), lse, None, None, C, 0, None, C,
                            scratch, N * 255, N, C, V)
    assert e.value.status == gk.GK_ERR_WORKSPACE


def test_softmax_ce_in_place(gkctx):
    from gpt_decoder_gb300 import gk

    torch = _t()
    rows, V = 64, 1000
    x = normal(810, rows, V)
    tg = synth.Stream(811).ints(rows, V)
    dx = dev(x)
    loss, lse = torch.zeros(1, device="cuda"), torch.empty(rows, device="cuda")
    gk.gk_softmax_ce_fwd(gkctx, dx, V, dev(tg), loss, lse, rows, V)
    gk.gk_softmax_ce_bwd(gkctx, dx, V, dev(tg), lse, None, dx, V, gk.GK_F32, rows, V)
    gk.gk_sync(gkctx)
    _, rlse = ops.softmax_ce_fwd(x, tg)
    assert_close(host(dx), ops.softmax_ce_bwd(x, tg, rlse, 1.0), 1e-5)


# ---------------------------------------------------------------------------- AdamW
@pytest.mark.parametrize("n", [1, 7, 4096 * 768 + 3])
def test_adamw(gkctx, n):
    from gpt_decoder_gb300 import gk

    torch = _t()
    p0, g, m0 = normal(900, n), normal(901, n), normal(902, n, std=0.1)
    v0 = np.abs(normal(903, n, std=0.1))
    p, dg, m, v = dev(p0), dev(g), dev(m0), dev(v0)
    pb = torch.empty(n, dtype=torch.bfloat16, device="cuda")
    for decay in (1, 0):
        p.copy_(dev(p0)); m.copy_(dev(m0)); v.copy_(dev(v0)); dg.copy_(dev(g))
        gk.gk_adamw_step(gkctx, [dict(p=p, g=dg, m=m, v=v, n=n, decay=decay, p_bf16=pb)], 3e-4, 0.9, 0.999, 1e-8,
                         0.01, 5, zero_grad=True)
        gk.gk_sync(gkctx)
        rp, rm, rv = ops.adamw(p0, g, m0, v0, 5, 3e-4, 0.9, 0.999, 1e-8, 0.01 if decay else 0.0)
        assert np.abs(host(p) - rp).max() <= 1e-6 * np.abs(rp).max()
        assert_close(host(m), rm, 1e-6)
        assert_close(host(v), rv, 1e-6)
        assert not host(dg).any()
        assert_close(host(pb), host(p), 5e-3)


# ------------------------------------------------------------------- split bf16
def _split(a):
    torch = _t()
    t = torch.as_tensor(np.asarray(a, dtype=np.float32))
    hi = t.to(torch.bfloat16)
    lo = (t - hi.float()).to(torch.bfloat16)
    return hi, lo


@pytest.mark.parametrize("N,K,M,transW", [(4096, 768, 3072, 0), (4096, 3072, 768, 0), (300, 96, 384, 0),
                                          (256, 256, 256, 1), (131, 64, 45, 0)])
@pytest.mark.parametrize("which", ["both", "W", "X"])
def test_matmul_fwd_split_bf16(gkctx, N, K, M, transW, which):
    """Split-bf16 operands (hi + lo planes, three products) track float32 operands closely."""
    from gpt_decoder_gb300 import gk

    torch = _t()
    x = normal(1100 + N, N, K)
    w = normal(1101 + K, M, K) if transW else normal(1101 + K, K, M)
    xh, xl = _split(x)
    wh, wl = _split(w)
    b = normal(1102, M)
    y = torch.empty(N, M, device="cuda")
    use_x, use_w = which in ("both", "X"), which in ("both", "W")
    gk.gk_matmul_fwd(gkctx, gk.GK_BF16, xh.cuda(), K, wh.cuda(), w.shape[1], transW, dev(b), None, 0, y, M, gk.GK_F32,
                     N, K, M, gk.GK_ACT_NONE, None, 0, xl.cuda() if use_x else None, wl.cuda() if use_w else None)
    gk.gk_sync(gkctx)
    xe = x if use_x else xh.float().numpy()
    we = w if use_w else wh.float().numpy()
    ref = (ops.matmul_t_fwd(xe, we) if transW else ops.matmul_fwd(xe, we)) + b
    # the dropped lo x lo term and the 16-bit pieces leave about 2^-16 relative error
    assert_close(host(y), ref, 1e-4)


def test_split_outputs_hold_the_float32_value(gkctx):
    """GK_BF16X2 outputs (GEMM with GELU, LayerNorm): hi + lo equals the float32 result."""
    from gpt_decoder_gb300 import gk

    torch = _t()
    N, K, M = 300, 96, 384
    x, w, b = normal(1200, N, K), normal(1201, K, M), normal(1202, M)
    y2 = torch.empty(2, N, M, dtype=torch.bfloat16, device="cuda")
    pre = torch.empty(N, M, dtype=torch.bfloat16, device="cuda")
    xh, xl = _split(x)
    wh, wl = _split(w)
    gk.gk_matmul_fwd(gkctx, gk.GK_BF16, xh.cuda(), K, wh.cuda(), M, 0, dev(b), None, 0, y2, M, gk.GK_BF16X2, N, K, M,
                     gk.GK_ACT_GELU, pre, M, xl.cuda(), wl.cuda())
    rows, C = 37, 768
    xx = normal(1203, rows, C) * 2 + 0.5
    gm, bt = normal(1204, C), normal(1205, C)
    ln2 = torch.empty(2, rows, C, dtype=torch.bfloat16, device="cuda")
    gk.gk_layernorm_fwd(gkctx, dev(xx), dev(gm), dev(bt), ln2, gk.GK_BF16X2, None, None, rows, C, 1e-5)
    gk.gk_sync(gkctx)
    ref = ops.gelu_fwd(ops.matmul_fwd(x, w) + b)
    got = y2[0].float().cpu().numpy() + y2[1].float().cpu().numpy()
    assert_close(got, ref, 1e-4)
    assert rel_l2(y2[0].float().cpu().numpy(), ref) > 1e-4  # the hi plane alone is bf16-coarse
    ry, _, _ = ops.layernorm_fwd(xx, gm, bt)
    got = ln2[0].float().cpu().numpy() + ln2[1].float().cpu().numpy()
    assert np.abs(got - ry).max() < 1e-5 * np.abs(ry).max()
