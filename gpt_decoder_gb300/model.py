"""GPT-2 training-step driver over libgk: buffers, and the gk_* calls in forward and reverse order.

The model is the pre-LN GPT-2 decoder of [LM4] ("Build a language model in C# from scratch
(4): running GPT-2 weights", "Loading weights into our classes"): embedding, L blocks of
x += attn_proj(attn(c_attn(ln_1(x)))), x += mlp_proj(gelu(c_fc(ln_2(x)))), then ln_f and
the tied head logits = ln_f(x) wte^T, softmax cross-entropy, and AdamW ([LM1] "Build a
language model in C# from scratch (1)", "The optimizer"). Parameters, gradients and AdamW
moments are single flat float32 buffers in libgk's layout (gk_gpt_offset), so AdamW is one
pass over two contiguous blocks (decayed matrices, undecayed vectors).

This module only allocates device memory (torch) and sequences calls; every arithmetic step
runs in libgk's kernels.

Modes: "fp32" runs every product on float32 operands (the faithful mode), by default as
3xTF32 on the tensor cores (math="3xtf32": each operand split into TF32 hi and lo parts, three
products accumulated in float32) or with math="fp32" as float32 FMA on the CUDA cores; "bf16"
keeps float32 master weights, moments, residual stream and logits, and feeds the matrix products bf16
operands (a bf16 weight copy that AdamW refreshes, bf16 activations) with float32
accumulation. In bf16 mode the forward products of the first `hi_layers` blocks (default 2)
use split-bf16 operands (value = hi + lo, two bf16 planes, three tensor-core products):
block 0's output is about ten times the embedding it is added to, so its operand rounding
sets the relative error of everything downstream. Measured on the GPT-2-124M shape, all-bf16
logits land at 0.021-0.022 max-abs from the float64 result; exact operands in the first two
blocks' products (their attention inputs and outputs still bf16) bring that to about 0.017.
Their backward is plain bf16 on the hi planes, like every other block.
"""
from __future__ import annotations

import torch

from . import gk

EPS = 1e-5


def pad_vocab(V: int, mult: int = 64) -> int:
    return (V + mult - 1) // mult * mult


class Gpt:
    def __init__(self, ctx: gk.Ctx, V, T, C, H, L, B, mode="fp32", device="cuda", hi_layers=2, fused_head=None,
                 math="3xtf32"):
        assert mode in ("fp32", "bf16")
        assert math in ("3xtf32", "fp32")
        self.ctx, self.mode, self.device = ctx, mode, device
        # arithmetic of the float32 products (the context's math mode, set before each pass)
        self.math = gk.GK_MATH_3XTF32 if math == "3xtf32" else gk.GK_MATH_FP32
        # bf16 mode: the LM head and the cross-entropy run fused (gk_lmhead_ce_*), with no
        # [N, V] logits tensor; fused_head=False keeps the separate head GEMM and CE kernels
        # (and self.logits) as in fp32 mode
        self.fused_head = (mode == "bf16") if fused_head is None else bool(fused_head)
        assert not self.fused_head or mode == "bf16", "the fused head takes bf16 operands"
        self.V, self.T, self.C, self.H, self.L, self.B = V, T, C, H, L, B
        self.hs = C // H
        self.N = B * T
        self.Vp = pad_vocab(V)
        self.cfg = gk.gk_gpt_cfg(V, T, C, H, L)
        self.numel = gk.gk_gpt_numel(self.cfg)
        self.n_decay = gk.gk_gpt_n_decay(self.cfg)
        f32 = dict(dtype=torch.float32, device=device)
        self.params = torch.zeros(self.numel, **f32)
        self.grads = torch.zeros(self.numel, **f32)
        self.m = torch.zeros(self.numel, **f32)
        self.v = torch.zeros(self.numel, **f32)
        self.dt = gk.GK_F32 if mode == "fp32" else gk.GK_BF16
        adt = torch.float32 if mode == "fp32" else torch.bfloat16
        self.params_bf16 = torch.zeros(self.numel, dtype=torch.bfloat16, device=device) if mode == "bf16" else None
        # low planes of the split-bf16 weights: the matrices of the first hi_layers blocks
        self.hi_lo = gk.gk_gpt_offset(self.cfg, gk.GK_T_ATTN_W, 0)
        self.hi_hi = self.hi_lo + min(hi_layers, L) * 12 * C * C if mode == "bf16" else self.hi_lo
        self.params_bf16_lo = (torch.zeros(max(1, self.hi_hi - self.hi_lo), dtype=torch.bfloat16, device=device)
                               if mode == "bf16" else None)
        self.step_count = 0
        N, C = self.N, C
        # per-block operand type of the products: float32 in fp32 mode, else bf16; in bf16 mode
        # the first hi_layers blocks' forward products take split-bf16 operands (hi + lo planes)
        self.ldt = [gk.GK_F32 if mode == "fp32" else gk.GK_BF16 for l in range(L)]
        self.split = [mode == "bf16" and l < hi_layers for l in range(L)]
        tdt = {gk.GK_F32: torch.float32, gk.GK_BF16: torch.bfloat16}

        def act(l, *shape, planes=1):
            if planes == 2 and self.split[l]:
                return torch.empty(2, *shape, dtype=torch.bfloat16, device=device)
            return torch.empty(*shape, dtype=tdt[self.ldt[l]], device=device)

        # residual stream: xs[2l] enters block l, xs[2l+1] is after its attention
        self.xs = [torch.empty(N, C, **f32) for _ in range(2 * L + 1)]
        self.ln1 = [act(l, N, C, planes=2) for l in range(L)]
        self.mu1 = [torch.empty(N, **f32) for _ in range(L)]
        self.rs1 = [torch.empty(N, **f32) for _ in range(L)]
        self.qkv = [act(l, N, 3 * C) for l in range(L)]
        self.y = [act(l, N, C) for l in range(L)]
        self.lse = [torch.empty(B * H * T, **f32) for _ in range(L)]
        self.ln2 = [act(l, N, C, planes=2) for l in range(L)]
        self.mu2 = [torch.empty(N, **f32) for _ in range(L)]
        self.rs2 = [torch.empty(N, **f32) for _ in range(L)]
        self.pre = [act(l, N, 4 * C) for l in range(L)]
        self.h = [act(l, N, 4 * C, planes=2) for l in range(L)]
        self.lnf = torch.empty(N, C, dtype=adt, device=device)
        self.muf = torch.empty(N, **f32)
        self.rsf = torch.empty(N, **f32)
        self.logits = None if self.fused_head else torch.empty(N, self.Vp, **f32)
        self.lse_ce = torch.empty(N, **f32)
        self.loss = torch.zeros(1, **f32)
        # backward buffers; with the fused head dlogits is the scratch for one vocabulary chunk
        # (up to 16384 columns, the chunks balanced)
        if self.fused_head:
            n_chunks = -(-V // 16384)
            self.head_chunk = -(-(-(-V // n_chunks)) // 256) * 256
            self.dlogits = torch.empty(N * self.head_chunk, dtype=torch.bfloat16, device=device)
        else:
            self.dlogits = torch.empty(N, self.Vp, dtype=adt, device=device)
        self.dx = torch.empty(N, C, **f32)
        self.dx_bf16 = torch.empty(N, C, dtype=torch.bfloat16, device=device) if mode == "bf16" else None
        self.dln = torch.empty(N, C, **f32)
        # per operand type: dpre / dy_attn share dmid; dqkv
        used = set(self.ldt)
        self.dmid = {d: torch.empty(N, 4 * C, dtype=tdt[d], device=device) for d in used}
        self.dqkv = {d: torch.empty(N, 3 * C, dtype=tdt[d], device=device) for d in used}

    # ------------------------------------------------------------ parameter access
    def off(self, which, layer=0):
        return gk.gk_gpt_offset(self.cfg, which, layer)

    def w(self, which, layer=0, for_gemm=False):
        """Address of a parameter tensor (the bf16 copy for GEMM operands in bf16 mode)."""
        o = self.off(which, layer)
        if for_gemm and self.mode == "bf16":
            return self.params_bf16.data_ptr() + 2 * o
        return self.params.data_ptr() + 4 * o

    def w_lo(self, which, layer):
        """Address of a block-weight matrix's low bf16 plane (split-bf16 blocks only)."""
        o = self.off(which, layer)
        assert self.hi_lo <= o < self.hi_hi
        return self.params_bf16_lo.data_ptr() + 2 * (o - self.hi_lo)

    def g(self, which, layer=0):
        return self.grads.data_ptr() + 4 * self.off(which, layer)

    TENSOR_NAMES = {
        gk.GK_T_LN1_W: "ln_1.weight", gk.GK_T_LN1_B: "ln_1.bias", gk.GK_T_ATTN_W: "attn.c_attn.weight",
        gk.GK_T_ATTN_B: "attn.c_attn.bias", gk.GK_T_ATTNPROJ_W: "attn.c_proj.weight",
        gk.GK_T_ATTNPROJ_B: "attn.c_proj.bias", gk.GK_T_LN2_W: "ln_2.weight", gk.GK_T_LN2_B: "ln_2.bias",
        gk.GK_T_FC_W: "mlp.c_fc.weight", gk.GK_T_FC_B: "mlp.c_fc.bias", gk.GK_T_MLPPROJ_W: "mlp.c_proj.weight",
        gk.GK_T_MLPPROJ_B: "mlp.c_proj.bias",
    }

    def named_slices(self, flat):
        """name -> view of `flat` (a tensor in the layout) for every parameter tensor."""
        C = self.C
        out = {"wte.weight": flat[self.off(gk.GK_T_WTE):][: self.V * C].view(self.V, C),
               "wpe.weight": flat[self.off(gk.GK_T_WPE):][: self.T * C].view(self.T, C),
               "ln_f.weight": flat[self.off(gk.GK_T_LNF_W):][:C], "ln_f.bias": flat[self.off(gk.GK_T_LNF_B):][:C]}
        shapes = {gk.GK_T_LN1_W: (C,), gk.GK_T_LN1_B: (C,), gk.GK_T_ATTN_W: (C, 3 * C), gk.GK_T_ATTN_B: (3 * C,),
                  gk.GK_T_ATTNPROJ_W: (C, C), gk.GK_T_ATTNPROJ_B: (C,), gk.GK_T_LN2_W: (C,), gk.GK_T_LN2_B: (C,),
                  gk.GK_T_FC_W: (C, 4 * C), gk.GK_T_FC_B: (4 * C,), gk.GK_T_MLPPROJ_W: (4 * C, C),
                  gk.GK_T_MLPPROJ_B: (C,)}
        for l in range(self.L):
            for which, name in self.TENSOR_NAMES.items():
                shp = shapes[which]
                n = 1
                for s in shp:
                    n *= s
                out[f"h.{l}.{name}"] = flat[self.off(which, l):][:n].view(*shp)
        return out

    def load(self, named):
        """Copy named float32 host arrays (GPT-2 checkpoint names) into the flat buffer."""
        views = self.named_slices(self.params)
        for k, v in named.items():
            views[k].copy_(torch.as_tensor(v, dtype=torch.float32))
        self.refresh_bf16()

    def refresh_bf16(self):
        """Recompute the bf16 operand copies (and low planes) from the float32 parameters."""
        if self.params_bf16 is not None:
            gk.gk_to_bf16(self.ctx, self.params, self.params_bf16, self.numel)
            n = self.hi_hi - self.hi_lo
            if n > 0:
                gk.gk_to_bf16(self.ctx, self.params.data_ptr() + 4 * self.hi_lo,
                              self.params_bf16.data_ptr() + 2 * self.hi_lo, n, y_lo=self.params_bf16_lo)

    # ------------------------------------------------------------- GEMM timing hook
    gemm_events = None  # a list: every matmul call appends (start event, end event, flops)

    def _timed(self, fn, args, flops):
        if self.gemm_events is None:
            return fn(*args)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        r = fn(*args)
        e1.record()
        self.gemm_events.append((e0, e1, flops))
        return r

    def _mm_fwd(self, *args):
        N, K, M = args[13:16]
        return self._timed(gk.gk_matmul_fwd, args, 2.0 * N * K * M)

    def _mm_bwd(self, *args):
        N, K, M = args[18:21]
        return self._timed(gk.gk_matmul_bwd, args, 4.0 * N * K * M)

    # ----------------------------------------------------------------- the step
    def forward(self, ids, targets):
        """Logits and loss of one batch (ids, targets: int32 device tensors [B*T])."""
        c, dt, N, C, H, hs, B, T = self.ctx, self.dt, self.N, self.C, self.H, self.hs, self.B, self.T
        gk.gk_set_math(c, self.math)
        gk.gk_embedding_fwd(c, ids, self.w(gk.GK_T_WTE), self.w(gk.GK_T_WPE), self.xs[0], B, T, C, self.V)
        for l in range(self.L):
            dt = self.ldt[l]
            bw = dt == gk.GK_BF16  # GEMM weights from the bf16 copy
            sp = self.split[l]
            lnd = gk.GK_BF16X2 if sp else dt  # LayerNorm / GELU outputs: two planes when split
            lo = (lambda buf: buf[1]) if sp else (lambda buf: None)
            wl = (lambda which: self.w_lo(which, l)) if sp else (lambda which: None)
            x_in, x_mid, x_out = self.xs[2 * l], self.xs[2 * l + 1], self.xs[2 * l + 2]
            # the LayerNorms also copy their input into the next residual buffer, which the
            # projection then adds into in place (a TMA reduce-add in the GEMM epilogue)
            gk.gk_layernorm_fwd(c, x_in, self.w(gk.GK_T_LN1_W, l), self.w(gk.GK_T_LN1_B, l), self.ln1[l], lnd,
                                self.mu1[l], self.rs1[l], N, C, EPS, x_copy=x_mid)
            self._mm_fwd(c, dt, self.ln1[l], C, self.w(gk.GK_T_ATTN_W, l, bw), 3 * C, 0,
                         self.w(gk.GK_T_ATTN_B, l), None, 0, self.qkv[l], 3 * C, dt, N, C, 3 * C,
                         gk.GK_ACT_NONE, None, 0, lo(self.ln1[l]), wl(gk.GK_T_ATTN_W))
            gk.gk_attn_fwd(c, dt, self.qkv[l], self.y[l], self.lse[l], B, T, H, hs)
            self._mm_fwd(c, dt, self.y[l], C, self.w(gk.GK_T_ATTNPROJ_W, l, bw), C, 0,
                         self.w(gk.GK_T_ATTNPROJ_B, l), x_mid, C, x_mid, C, gk.GK_F32, N, C, C,
                         gk.GK_ACT_NONE, None, 0, None, wl(gk.GK_T_ATTNPROJ_W))
            gk.gk_layernorm_fwd(c, x_mid, self.w(gk.GK_T_LN2_W, l), self.w(gk.GK_T_LN2_B, l), self.ln2[l], lnd,
                                self.mu2[l], self.rs2[l], N, C, EPS, x_copy=x_out)
            self._mm_fwd(c, dt, self.ln2[l], C, self.w(gk.GK_T_FC_W, l, bw), 4 * C, 0,
                         self.w(gk.GK_T_FC_B, l), None, 0, self.h[l], 4 * C, lnd, N, C, 4 * C,
                         gk.GK_ACT_GELU, self.pre[l], 4 * C, lo(self.ln2[l]), wl(gk.GK_T_FC_W))
            self._mm_fwd(c, dt, self.h[l], 4 * C, self.w(gk.GK_T_MLPPROJ_W, l, bw), C, 0,
                         self.w(gk.GK_T_MLPPROJ_B, l), x_out, C, x_out, C, gk.GK_F32, N, 4 * C, C,
                         gk.GK_ACT_NONE, None, 0, lo(self.h[l]), wl(gk.GK_T_MLPPROJ_W))
        gk.gk_layernorm_fwd(c, self.xs[-1], self.w(gk.GK_T_LNF_W), self.w(gk.GK_T_LNF_B), self.lnf, self.dt, self.muf,
                            self.rsf, N, C, EPS)
        if self.fused_head:
            self._timed(gk.gk_lmhead_ce_fwd, (c, self.dt, self.lnf, C, self.w(gk.GK_T_WTE, 0, True), C, targets,
                                              self.loss, self.lse_ce, N, C, self.V), 2.0 * N * C * self.V)
            return self.loss
        self._mm_fwd(c, self.dt, self.lnf, C, self.w(gk.GK_T_WTE, 0, True), C, 1, None, None, 0, self.logits,
                         self.Vp, gk.GK_F32, N, C, self.V)
        gk.gk_softmax_ce_fwd(c, self.logits, self.Vp, targets, self.loss, self.lse_ce, N, self.V)
        return self.loss

    def backward(self, ids, targets):
        """Parameter gradients ADDED into self.grads (zero them first, or let AdamW do it)."""
        c, dt, N, C, H, hs, B, T = self.ctx, self.dt, self.N, self.C, self.H, self.hs, self.B, self.T
        gk.gk_set_math(c, self.math)
        if self.fused_head:
            # dlnf = dlogits wte, dwte += dlogits^T lnf, the logits recomputed per vocabulary chunk
            # (the timed FLOPs count the two products only)
            self._timed(gk.gk_lmhead_ce_bwd, (c, self.dt, self.lnf, C, self.w(gk.GK_T_WTE, 0, True), C, targets,
                                              self.lse_ce, None, self.dln, C, 0, self.g(gk.GK_T_WTE), C,
                                              self.dlogits, self.dlogits.numel(), N, C, self.V),
                        4.0 * N * C * self.V)
        else:
            gk.gk_softmax_ce_bwd(c, self.logits, self.Vp, targets, self.lse_ce, None, self.dlogits, self.Vp, self.dt,
                                 N, self.V)
            # tied head: dlnf = dlogits wte; dwte += dlogits^T lnf
            self._mm_bwd(c, self.dt, self.lnf, C, self.w(gk.GK_T_WTE, 0, True), C, 1, self.dlogits, self.Vp, self.dln,
                         C, gk.GK_F32, 0, None, 0, self.g(gk.GK_T_WTE), C, None, N, C, self.V)
        # the LayerNorm backwards also leave the column sums of the residual gradient they
        # produce: the bias gradients of the projections whose output gradient it is
        gk.gk_layernorm_bwd(c, self.xs[-1], self.w(gk.GK_T_LNF_W), self.muf, self.rsf, self.dln, self.dx, 0,
                            self.dx_bf16, self.g(gk.GK_T_LNF_W), self.g(gk.GK_T_LNF_B), N, C,
                            dx_colsum=self.g(gk.GK_T_MLPPROJ_B, self.L - 1))
        for l in reversed(range(self.L)):
            dt = self.ldt[l]
            bw = dt == gk.GK_BF16
            dxg = self.dx_bf16 if bw else self.dx  # the residual gradient as this block's GEMM operand
            x_in, x_mid = self.xs[2 * l], self.xs[2 * l + 1]
            hi = (lambda buf: buf[0]) if self.split[l] else (lambda buf: buf)  # bf16 plane of split buffers
            dpre = self.dmid[dt]
            # x_out = x_mid + h Wp + bp   (GELU backward fused into the dX product)
            self._mm_bwd(c, dt, hi(self.h[l]), 4 * C, self.w(gk.GK_T_MLPPROJ_W, l, bw), C, 0, dxg, C, dpre,
                             4 * C, dt, 0, self.pre[l], 4 * C, self.g(gk.GK_T_MLPPROJ_W, l), C,
                             None, N, 4 * C, C)
            self._mm_bwd(c, dt, hi(self.ln2[l]), C, self.w(gk.GK_T_FC_W, l, bw), 4 * C, 0, dpre, 4 * C, self.dln,
                             C, gk.GK_F32, 0, None, 0, self.g(gk.GK_T_FC_W, l), 4 * C, self.g(gk.GK_T_FC_B, l), N,
                             C, 4 * C)
            gk.gk_layernorm_bwd(c, x_mid, self.w(gk.GK_T_LN2_W, l), self.mu2[l], self.rs2[l], self.dln, self.dx, 1,
                                self.dx_bf16, self.g(gk.GK_T_LN2_W, l), self.g(gk.GK_T_LN2_B, l), N, C,
                                dx_colsum=self.g(gk.GK_T_ATTNPROJ_B, l))
            # x_mid = x_in + y Wo + bo
            dy = self.dmid[dt]
            self._mm_bwd(c, dt, self.y[l], C, self.w(gk.GK_T_ATTNPROJ_W, l, bw), C, 0, dxg, C, dy, C, dt, 0,
                             None, 0, self.g(gk.GK_T_ATTNPROJ_W, l), C, None, N, C, C)
            gk.gk_attn_bwd(c, dt, self.qkv[l], self.y[l], self.lse[l], dy, self.dqkv[dt], B, T, H, hs)
            self._mm_bwd(c, dt, hi(self.ln1[l]), C, self.w(gk.GK_T_ATTN_W, l, bw), 3 * C, 0, self.dqkv[dt], 3 * C,
                             self.dln, C, gk.GK_F32, 0, None, 0, self.g(gk.GK_T_ATTN_W, l), 3 * C,
                             self.g(gk.GK_T_ATTN_B, l), N, C, 3 * C)
            gk.gk_layernorm_bwd(c, x_in, self.w(gk.GK_T_LN1_W, l), self.mu1[l], self.rs1[l], self.dln, self.dx, 1,
                                self.dx_bf16, self.g(gk.GK_T_LN1_W, l), self.g(gk.GK_T_LN1_B, l), N, C,
                                dx_colsum=self.g(gk.GK_T_MLPPROJ_B, l - 1) if l > 0 else None)
        gk.gk_embedding_bwd(c, ids, self.dx, self.g(gk.GK_T_WTE), self.g(gk.GK_T_WPE), B, T, C, self.V)

    def adamw_cuts(self):
        """(start, end, decay, writes low plane) spans of the flat buffer for AdamW: decayed
        matrices (the split-bf16 blocks' matrices also refresh their low planes), then the
        undecayed vectors."""
        cuts = [(0, self.hi_lo, 1, False), (self.hi_lo, self.hi_hi, 1, True), (self.hi_hi, self.n_decay, 1, False),
                (self.n_decay, self.numel, 0, False)]
        return [c for c in cuts if c[1] > c[0]]

    def adamw(self, lr, beta1=0.9, beta2=0.999, eps=1e-8, wd=0.0, zero_grad=True):
        self.step_count += 1
        pb = self.params_bf16
        P, G, M_, V_ = (t.data_ptr() for t in (self.params, self.grads, self.m, self.v))

        def blk(a, b, decay, with_lo=False):
            return dict(p=P + 4 * a, g=G + 4 * a, m=M_ + 4 * a, v=V_ + 4 * a, n=b - a, decay=decay,
                        p_bf16=None if pb is None else pb.data_ptr() + 2 * a,
                        p_bf16_lo=self.params_bf16_lo.data_ptr() + 2 * (a - self.hi_lo) if with_lo else None)

        blocks = [blk(a, b, d, lo) for (a, b, d, lo) in self.adamw_cuts()]
        gk.gk_adamw_step(self.ctx, blocks, lr, beta1, beta2, eps, wd, self.step_count, zero_grad)

    def train_step(self, ids, targets, lr, wd, beta1=0.9, beta2=0.999, eps=1e-8):
        """One fwd + bwd + AdamW step; gradients are zeroed inside AdamW for the next step."""
        loss = self.forward(ids, targets)
        self.backward(ids, targets)
        self.adamw(lr, beta1, beta2, eps, wd, zero_grad=True)
        return loss
