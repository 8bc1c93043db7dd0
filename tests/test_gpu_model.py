"""Whole training-step parity (forward, backward, AdamW) of the libgk driver against the oracle.

Workloads: the tiny character model (V=64, T=64, C=96, H=4, L=4, B=8, seed 0), a ragged shape
and the GPT-2-124M shape (B=4, T=1024, seed 2), each in fp32, bf16 with the separate LM head and
CE kernels, and bf16 with the fused LM head + CE (no logits tensor: loss, gradients, update). Tolerances: faithful (fp32)
logits max-abs <= 5e-4, gradient relative-L2 <= 1e-4 per tensor; fast (bf16) logits
max-abs <= 2e-2, gradient relative-L2 <= 1e-2.
"""
import numpy as np
import pytest

import synth
from oracle import gpt as ogpt
from tests.conftest import rel_l2

pytestmark = pytest.mark.gpu

TOL = {"fp32": dict(logits=5e-4, grad=1e-4), "fp32-fma": dict(logits=5e-4, grad=1e-4),
       "bf16": dict(logits=2e-2, grad=1e-2), "bf16-fused": dict(logits=2e-2, grad=1e-2)}
# "fp32": the faithful mode's float32 products as 3xTF32 on the tensor cores; "fp32-fma": the
# same mode with float32 FMA on the CUDA cores
MODES = ["fp32", "fp32-fma", "bf16", "bf16-fused"]
LR, WD = 3e-4, 0.01


def _run_step(gkctx, s, B, seed, mode):
    import torch

    from gpt_decoder_gb300.model import Gpt

    ids, targets, params = synth.training_case(s, B, seed)
    # "bf16-fused": the fused LM head + cross-entropy (no logits tensor); "bf16": the separate
    # head GEMM and CE kernels, whose logits are checked
    m = Gpt(gkctx, s.V, s.T, s.C, s.H, s.L, B, mode=mode.split("-")[0], fused_head=mode == "bf16-fused",
            math="fp32" if mode == "fp32-fma" else "3xtf32")
    m.load(params)
    d_ids = torch.as_tensor(ids.reshape(-1)).cuda()
    d_tg = torch.as_tensor(targets.reshape(-1)).cuda()
    loss = m.forward(d_ids, d_tg)
    logits = None if m.logits is None else m.logits[:, : s.V].cpu().numpy()
    m.backward(d_ids, d_tg)
    from gpt_decoder_gb300 import gk

    gk.gk_sync(gkctx)
    grads = {k: v.cpu().numpy() for k, v in m.named_slices(m.grads).items()}
    m.adamw(LR, wd=WD, zero_grad=True)
    gk.gk_sync(gkctx)
    newp = {k: v.cpu().numpy() for k, v in m.named_slices(m.params).items()}
    assert not m.grads.any().item(), "AdamW's fused ZeroGrad left a gradient"
    return dict(loss=loss.item(), logits=logits, grads=grads, params=newp, inputs=(ids, targets, params))


def _oracle(s, inputs):
    ids, targets, params = inputs
    sh = ogpt.Shape(s.V, s.T, s.C, s.H, s.L)
    loss, grads, logits, _ = ogpt.loss_and_grads(params, ids, targets, sh)
    newp, _ = ogpt.adamw_step(params, grads, {}, 1, LR, wd=WD)
    return dict(loss=loss, logits=logits, grads=grads, params=newp)


def _compare(got, ref, mode):
    tol = TOL[mode]
    assert abs(got["loss"] - ref["loss"]) < tol["logits"], (got["loss"], ref["loss"])
    if got["logits"] is not None:
        assert np.abs(got["logits"] - ref["logits"]).max() <= tol["logits"]
    worst = max((rel_l2(got["grads"][k], ref["grads"][k]), k) for k in ref["grads"])
    assert worst[0] <= tol["grad"], worst
    # AdamW after one step: m_hat / sqrt(v_hat) = g / (|g| + eps), i.e. the sign of g once
    # |g| >> eps, so an element whose gradient error is comparable to the gradient itself can
    # move by 2 lr either way. The update is checked on elements whose gradient is clear:
    # |g_ref| above 10x this element's own gradient error and above 100x AdamW's eps; the
    # others are counted.
    flips = 0
    for k, p in ref["params"].items():
        g = ref["grads"][k]
        clear = (np.abs(g) > 10 * np.abs(got["grads"][k] - g)) & (np.abs(g) > 100 * 1e-8)
        d = np.abs(got["params"][k] - p)
        assert d[clear].max(initial=0.0) <= 1e-6 + 1e-3 * LR + 1e-6 * np.abs(p[clear]).max(initial=0.0), k
        flips += int((d[~clear] > 1e-3 * LR).sum())
    return worst, flips


@pytest.mark.parametrize("mode", MODES)
def test_tiny_training_step(gkctx, mode):
    s = synth.TINY
    got = _run_step(gkctx, s, 8, 0, mode)
    ref = _oracle(s, got["inputs"])
    worst, flips = _compare(got, ref, mode)
    print(f"tiny {mode}: loss {got['loss']:.6f} vs {ref['loss']:.6f}; worst grad rel-L2 {worst}; "
          f"small-gradient sign flips {flips}")


@pytest.mark.parametrize("mode", MODES)
def test_ragged_shapes_step(gkctx, mode):
    # vocabulary, context and width that leave partial tiles everywhere
    s = synth.GptShape(V=50, T=37, C=64, H=2, L=2)
    got = _run_step(gkctx, s, 3, 11, mode)
    ref = _oracle(s, got["inputs"])
    _compare(got, ref, mode)


_GPT2_ORACLE = {}


@pytest.mark.slow
@pytest.mark.parametrize("mode", MODES)
def test_gpt2_124m_training_step(gkctx, mode):
    s = synth.GPT2_124M
    got = _run_step(gkctx, s, 4, 2, mode)
    if "ref" not in _GPT2_ORACLE:
        _GPT2_ORACLE["ref"] = _oracle(s, got["inputs"])
    ref = _GPT2_ORACLE["ref"]
    worst, flips = _compare(got, ref, mode)
    dl = "n/a" if got["logits"] is None else f"{np.abs(got['logits'] - ref['logits']).max():.3e}"
    print(f"gpt2 {mode}: loss {got['loss']:.6f} vs {ref['loss']:.6f}; max |dlogits| {dl}; worst grad {worst}; "
          f"flips {flips}")


def test_loss_decreases_over_steps(gkctx):
    import torch

    from gpt_decoder_gb300 import gk
    from gpt_decoder_gb300.model import Gpt

    s = synth.TINY
    ids, targets, params = synth.training_case(s, 8, 0)
    m = Gpt(gkctx, s.V, s.T, s.C, s.H, s.L, 8, mode="bf16")
    m.load(params)
    d_ids = torch.as_tensor(ids.reshape(-1)).cuda()
    d_tg = torch.as_tensor(targets.reshape(-1)).cuda()
    losses = []
    for _ in range(20):
        losses.append(m.train_step(d_ids, d_tg, 1e-3, 0.01).item())
    gk.gk_sync(gkctx)
    assert losses[-1] < losses[0] - 0.3, losses


def test_bench_batch_forward_equals_its_four_quarters(gkctx):
    """bench.py's configuration (GPT-2-124M, B=16 x T=1024, bf16 with the fused head): rows do
    not interact in the forward, and every forward kernel reduces within a row in an order that
    does not depend on the batch, so the B=16 launches (their tile counts, CTA-pair grids) must
    leave every row's residual stream and log-sum-exp bit-identical to those of the four B=4
    quarters, and the loss equal to the mean of the quarters' losses up to float32 rounding.
    (The backward is checked against the oracle at B=16 below: there, float32 reductions whose
    order depends on the launch shape, re-rounded to bf16 at every block, make B=16 and B=4
    differ at the bf16 error level, not bit for bit.)"""
    import torch

    from gpt_decoder_gb300 import gk
    from gpt_decoder_gb300.model import Gpt

    s = synth.GPT2_124M
    ids, targets, params = synth.training_case(s, 16, 2)
    dev = lambda a: torch.as_tensor(np.ascontiguousarray(a).reshape(-1)).cuda()
    m16 = Gpt(gkctx, s.V, s.T, s.C, s.H, s.L, 16, mode="bf16")
    m16.load(params)
    loss16 = float(m16.forward(dev(ids), dev(targets)).item())
    keep = {f"xs{i}": m16.xs[i].clone() for i in range(1, len(m16.xs))}
    keep["lse"] = m16.lse_ce.clone()
    del m16
    m4 = Gpt(gkctx, s.V, s.T, s.C, s.H, s.L, 4, mode="bf16")
    m4.load(params)
    losses = []
    n = 4 * s.T
    for k in range(4):
        q = slice(4 * k, 4 * k + 4)
        losses.append(float(m4.forward(dev(ids[q]), dev(targets[q])).item()))
        gk.gk_sync(gkctx)
        for name, full in keep.items():
            part = m4.lse_ce if name == "lse" else m4.xs[int(name[2:])]
            assert torch.equal(full[k * n:(k + 1) * n], part), (k, name)
    assert abs(loss16 - sum(losses) / 4) < 1e-5, (loss16, losses)


_GPT2_B16_ORACLE = {}


@pytest.mark.slow
def test_gpt2_124m_bench_config_step_vs_oracle(gkctx):
    """The step bench.py times (GPT-2-124M, B=16 x T=1024, bf16 with the fused LM head) against
    the oracle at the fast-mode tolerances: loss, per-tensor gradient relative-L2 and the AdamW
    update. The oracle's B=16 gradient is the mean of its four B=4 quarters' gradients (float64;
    the loss is a mean over rows, so this is the same quantity), which keeps its host memory at
    the B=4 size."""
    s = synth.GPT2_124M
    got = _run_step(gkctx, s, 16, 2, "bf16-fused")
    if "ref" not in _GPT2_B16_ORACLE:
        ids, targets, params = got["inputs"]
        sh = ogpt.Shape(s.V, s.T, s.C, s.H, s.L)
        loss, grads = 0.0, None
        for k in range(4):
            q = slice(4 * k, 4 * k + 4)
            lq, gq, _, _ = ogpt.loss_and_grads(params, ids[q], targets[q], sh)
            loss += lq / 4
            grads = {n: v / 4 for n, v in gq.items()} if grads is None else {n: grads[n] + gq[n] / 4 for n in grads}
        newp, _ = ogpt.adamw_step(params, grads, {}, 1, LR, wd=WD)
        _GPT2_B16_ORACLE["ref"] = dict(loss=loss, logits=None, grads=grads, params=newp)
    ref = _GPT2_B16_ORACLE["ref"]
    worst, flips = _compare(got, ref, "bf16-fused")
    print(f"gpt2 B=16 bf16-fused: loss {got['loss']:.6f} vs {ref['loss']:.6f}; worst grad {worst}; flips {flips}")
