"""KV-cache decode parity: prefill, decode steps and token selection against the oracle.

Greedy ids are compared teacher-forced: both sides are fed the oracle's token at every step,
and a step passes if the ids agree or the oracle's top-2 gap is below twice the measured
logit error (a near-tie, reported, not failed). Top-k selection is checked bit-exactly by
running the oracle's selection on the GPU's own logits with the same Philox draw.
"""
import numpy as np
import pytest

import synth
from oracle import gpt as ogpt
from oracle import sampling

pytestmark = pytest.mark.gpu


def _setup(gkctx, s, B, Tp, seed, Tmax):
    import torch

    from gpt_decoder_gb300 import gk
    from gpt_decoder_gb300.model import Gpt

    prompt, params = synth.prompt_case(s, B, Tp, seed)
    m = Gpt(gkctx, s.V, s.T, s.C, s.H, s.L, 1, mode="fp32")  # holds the flat parameters
    m.load(params)
    kv = gk.KvCache(gkctx, m.cfg, B, Tmax)
    return prompt, params, m, kv


def _teacher_forced(gkctx, s, B, Tp, n_steps, seed):
    import torch

    from gpt_decoder_gb300 import gk

    prompt, params, m, kv = _setup(gkctx, s, B, Tp, seed, Tp + n_steps)
    sh = ogpt.Shape(s.V, s.T, s.C, s.H, s.L)
    # the oracle's greedy continuation, then both sides fed those tokens
    picks, ologits = ogpt.generate(params, prompt, n_steps, sh, top_k=1)
    logits = torch.empty(B, s.V, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    gk.gk_prefill(gkctx, m.params, kv, torch.as_tensor(prompt.reshape(-1)).cuda(), Tp, logits)
    gk.gk_sample(gkctx, kv, logits, s.V, nxt, None)
    got_logits, got_ids = [logits.cpu().numpy()], [nxt.cpu().numpy()]
    for i in range(n_steps):
        feed = torch.as_tensor(picks[i].astype(np.int32)).cuda()
        gk.gk_decode_step(gkctx, m.params, kv, feed, logits, nxt, None)
        got_logits.append(logits.cpu().numpy())
        got_ids.append(nxt.cpu().numpy())
    gk.gk_sync(gkctx)
    assert kv.length() == Tp + n_steps
    got_logits, got_ids = np.array(got_logits), np.array(got_ids)
    err = np.abs(got_logits - ologits).max()
    srt = np.sort(ologits, axis=-1)
    gap = srt[..., -1] - srt[..., -2]
    mismatch = got_ids != picks
    near = mismatch & (gap < 2 * err)
    kv.close()
    return err, int(mismatch.sum()), int(near.sum()), got_ids, picks


@pytest.mark.parametrize("B", [1, 2, 4, 8])  # 8: the batch-8 GEMVs and LM head of the per-layer launches
def test_tiny_decode_teacher_forced(gkctx, B):
    err, mism, near, _, _ = _teacher_forced(gkctx, synth.TINY, B, 20, 40, 3)
    assert err <= 5e-4
    assert mism == near, (mism, near)


@pytest.mark.slow
@pytest.mark.parametrize("B", [1, 16])
def test_gpt2_decode_teacher_forced(gkctx, B):
    err, mism, near, _, _ = _teacher_forced(gkctx, synth.GPT2_124M, B, 512, 256, 3)
    print(f"gpt2 decode B={B}: max |logit diff| {err:.3e}, mismatched ids {mism}, near-ties {near}")
    assert err <= 5e-4
    assert mism == near


@pytest.mark.parametrize("sample", [None, (5, 0.8, 11, 3)])
@pytest.mark.parametrize("B", [2, 3])  # the persistent step, the per-layer launches
def test_decode_run_matches_step_by_step(gkctx, sample, B):
    """gk_decode_run (one captured step replayed as a graph) gives bit-identical logits,
    selections and cache to gk_decode_step called step by step, across two runs (the second
    replays the same graph), with tokens and next as one buffer or two."""
    import torch

    from gpt_decoder_gb300 import gk

    s, Tp, n1, n2 = synth.TINY, 9, 6, 5
    stream = torch.cuda.Stream()
    ctx = gk.Ctx(stream, 64 << 20)
    outs = []
    for path in ("steps", "run-shared", "run-separate"):
        prompt, params, m, kv = _setup(ctx, s, B, Tp, 7, Tp + n1 + n2)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            logits = torch.empty(B, s.V, device="cuda")
            tok = torch.empty(B, dtype=torch.int32, device="cuda")
            gk.gk_prefill(ctx, m.params, kv, torch.as_tensor(prompt.reshape(-1)).cuda(), Tp, logits)
            gk.gk_sample(ctx, kv, logits, s.V, tok, sample)
            seen = []
            if path == "steps":
                for i in range(n1 + n2):
                    gk.gk_decode_step(ctx, m.params, kv, tok, logits, tok, sample)
                    seen.append(tok.clone())
            else:
                nxt = tok if path == "run-shared" else torch.empty_like(tok)
                for n in (n1, n2):
                    gk.gk_decode_run(ctx, m.params, kv, tok, logits, nxt, n, sample)
                    seen.append(nxt.clone())
        gk.gk_sync(ctx)
        assert kv.length() == Tp + n1 + n2
        outs.append((logits.cpu().numpy(), tok.cpu().numpy(), [t.cpu().numpy() for t in seen]))
        kv.close()
    ref_logits, ref_tok, ref_seen = outs[0]
    for got_logits, got_tok, got_seen in outs[1:]:
        assert np.array_equal(got_logits, ref_logits)
        assert np.array_equal(got_tok, ref_tok)
        assert np.array_equal(got_seen[0], ref_seen[n1 - 1]) and np.array_equal(got_seen[1], ref_seen[-1])
    ctx.close()


def test_decode_run_overflow_runs_nothing(gkctx):
    import torch

    from gpt_decoder_gb300 import gk

    s, B, Tp = synth.TINY, 2, 5
    prompt, params, m, kv = _setup(gkctx, s, B, Tp, 7, Tp + 3)
    logits = torch.empty(B, s.V, device="cuda")
    tok = torch.zeros(B, dtype=torch.int32, device="cuda")
    gk.gk_prefill(gkctx, m.params, kv, torch.as_tensor(prompt.reshape(-1)).cuda(), Tp, logits)
    with pytest.raises(gk.GkError) as e:
        gk.gk_decode_run(gkctx, m.params, kv, tok, logits, tok, 4)
    assert e.value.status == gk.GK_ERR_OVERFLOW
    assert kv.length() == Tp
    gk.gk_decode_run(gkctx, m.params, kv, tok, logits, tok, 3)
    gk.gk_sync(gkctx)
    assert kv.length() == Tp + 3
    kv.close()


def test_cached_decode_equals_training_forward(gkctx):
    """The GPU's cached path reproduces its own full causal forward (fp32)."""
    import torch

    from gpt_decoder_gb300 import gk
    from gpt_decoder_gb300.model import Gpt

    s = synth.GptShape(V=64, T=32, C=96, H=4, L=2)
    B, Tp, n = 2, 10, 12
    prompt, params = synth.prompt_case(s, B, Tp + n, 5)
    full = Gpt(gkctx, s.V, s.T, s.C, s.H, s.L, B, mode="fp32")
    full.load(params)
    ids = np.zeros((B, s.T), np.int32)
    ids[:, : Tp + n] = prompt
    d_ids = torch.as_tensor(ids.reshape(-1)).cuda()
    full.forward(d_ids, d_ids)
    ref = full.logits[:, : s.V].reshape(B, s.T, s.V).cpu().numpy()
    kv = gk.KvCache(gkctx, full.cfg, B, Tp + n)
    logits = torch.empty(B, s.V, device="cuda")
    gk.gk_prefill(gkctx, full.params, kv, torch.as_tensor(prompt[:, :Tp].reshape(-1).copy()).cuda(), Tp, logits)
    worst = np.abs(logits.cpu().numpy() - ref[:, Tp - 1]).max()
    for i in range(n):
        tok = torch.as_tensor(prompt[:, Tp + i].copy()).cuda()
        gk.gk_decode_step(gkctx, full.params, kv, tok, logits, None, None)
        worst = max(worst, np.abs(logits.cpu().numpy() - ref[:, Tp + i]).max())
    gk.gk_sync(gkctx)
    assert worst < 1e-4
    with pytest.raises(gk.GkError) as e:
        gk.gk_decode_step(gkctx, full.params, kv, tok, logits, None, None)
    assert e.value.status == gk.GK_ERR_OVERFLOW
    kv.close()


@pytest.mark.parametrize("top_k,temp", [(40, 1.0), (3, 0.7), (0, 1.0), (64, 2.0)])
def test_topk_selection_matches_oracle_on_gpu_logits(gkctx, top_k, temp):
    import torch

    from gpt_decoder_gb300 import gk

    s = synth.TINY
    B = 4
    prompt, params, m, kv = _setup(gkctx, s, B, 8, 9, 40)
    logits = torch.empty(B, s.V, device="cuda")
    nxt = torch.empty(B, dtype=torch.int32, device="cuda")
    gk.gk_prefill(gkctx, m.params, kv, torch.as_tensor(prompt.reshape(-1)).cuda(), 8, logits)
    seed, counter = 4, 100
    for step in range(30):
        gk.gk_decode_step(gkctx, m.params, kv, nxt if step else torch.as_tensor(prompt[:, -1].copy()).cuda(), logits,
                          nxt, (top_k, temp, seed, counter))
        lg = logits.cpu().numpy()
        got = nxt.cpu().numpy()
        for b in range(B):
            # this selection's index is `step` (prefill made none)
            u = sampling.uniform(seed, counter + step, b)
            want = sampling.topk_sample(lg[b].astype(np.float64), top_k, temp, u)
            assert got[b] == want, (step, b, got[b], want)
    gk.gk_sync(gkctx)
    kv.close()


def test_topk_ties_are_kept_and_greedy_takes_lowest_index(gkctx):
    import torch

    from gpt_decoder_gb300 import gk

    s = synth.GptShape(V=10, T=8, C=8, H=2, L=1)
    cfg = gk.gk_gpt_cfg(s.V, s.T, s.C, s.H, s.L)
    kv = gk.KvCache(gkctx, cfg, 3, 4)
    row = np.array([0.5, 2.0, 1.0, 2.0, 1.0, 1.0, -3.0, 0.0, 1.0, -1.0], np.float32)
    lg = torch.as_tensor(np.stack([row] * 3)).cuda()
    nxt = torch.empty(3, dtype=torch.int32, device="cuda")
    gk.gk_sample(gkctx, kv, lg, s.V, nxt, None)
    assert list(nxt.cpu().numpy()) == [1, 1, 1]
    for sel in range(40):
        gk.gk_sample(gkctx, kv, lg, s.V, nxt, (3, 1.0, 11, 0))
        got = nxt.cpu().numpy()
        for b in range(3):
            u = sampling.uniform(11, sel + 1, b)
            assert got[b] == sampling.topk_sample(row, 3, 1.0, u)
            assert row[got[b]] >= 1.0
    gk.gk_sync(gkctx)
    kv.close()


def _uncached(gkctx, s, B, Tp, n_new, seed, sample):
    import torch

    from gpt_decoder_gb300 import gk

    prompt, params, m, kv = _setup(gkctx, s, B, Tp, seed, Tp + n_new)
    ids = torch.zeros(B, Tp + n_new, dtype=torch.int32, device="cuda")
    ids[:, :Tp] = torch.as_tensor(prompt.reshape(B, Tp))
    logits = torch.empty(B, s.V, device="cuda")
    gk.gk_generate_uncached(gkctx, m.params, kv, ids, Tp, n_new, logits, sample)
    gk.gk_sync(gkctx)
    out = ids.cpu().numpy()
    kv.close()
    return prompt, params, m, out


@pytest.mark.parametrize("B", [1, 3])
def test_uncached_generate_matches_oracle_greedy(gkctx, B):
    """[LM4] Generate (a full forward per token): the prompt columns are left alone and each
    row's greedy continuation is the oracle's up to its first near-tie."""
    s, Tp, n = synth.TINY, 12, 16
    prompt, params, _, out = _uncached(gkctx, s, B, Tp, n + 1, 5, None)
    assert np.array_equal(out[:, :Tp], prompt.reshape(B, Tp))
    picks, ologits = ogpt.generate(params, prompt, n, ogpt.Shape(s.V, s.T, s.C, s.H, s.L), top_k=1)
    got = out[:, Tp:].T  # [n + 1, B], like picks
    srt = np.sort(ologits, axis=-1)
    gap = srt[..., -1] - srt[..., -2]
    for b in range(B):
        bad = np.nonzero(got[:, b] != picks[:, b])[0]
        if len(bad):
            j = bad[0]
            assert gap[j, b] < 1e-3, (b, j, gap[j, b])


@pytest.mark.parametrize("sample", [None, (5, 0.8, 11, 3)])
def test_uncached_generate_equals_cached_loop(gkctx, sample):
    """Uncached and cached generation select the same tokens with the same draws: selection i
    of the uncached loop uses the counter the cached loop gives its i-th selection."""
    import torch

    from gpt_decoder_gb300 import gk

    s, B, Tp, n = synth.TINY, 2, 10, 12
    _, _, _, out = _uncached(gkctx, s, B, Tp, n + 1, 9, sample)
    prompt, params, m, kv = _setup(gkctx, s, B, Tp, 9, Tp + n)
    logits = torch.empty(B, s.V, device="cuda")
    tok = torch.empty(B, dtype=torch.int32, device="cuda")
    gk.gk_prefill(gkctx, m.params, kv, torch.as_tensor(prompt.reshape(-1)).cuda(), Tp, logits)
    gk.gk_sample(gkctx, kv, logits, s.V, tok, sample)
    seen = [tok.cpu().numpy()]
    for _ in range(n):
        gk.gk_decode_step(gkctx, m.params, kv, tok, logits, tok, sample)
        seen.append(tok.cpu().numpy())
    gk.gk_sync(gkctx)
    kv.close()
    assert np.array_equal(out[:, Tp:].T, np.array(seen))


def test_uncached_generate_overflow_runs_nothing(gkctx):
    import torch

    from gpt_decoder_gb300 import gk

    s, B, Tp = synth.TINY, 2, 5
    prompt, params, m, kv = _setup(gkctx, s, B, Tp, 7, Tp + 3)
    ids = torch.full((B, Tp + 5), -1, dtype=torch.int32, device="cuda")
    ids[:, :Tp] = torch.as_tensor(prompt.reshape(B, Tp))
    logits = torch.empty(B, s.V, device="cuda")
    with pytest.raises(gk.GkError) as e:
        gk.gk_generate_uncached(gkctx, m.params, kv, ids, Tp, 5, logits)
    assert e.value.status == gk.GK_ERR_OVERFLOW
    assert (ids[:, Tp:].cpu().numpy() == -1).all()
    ids4 = ids[:, :Tp + 4].contiguous()  # row stride Tp + n_new
    gk.gk_generate_uncached(gkctx, m.params, kv, ids4, Tp, 4, logits)  # Tp + 3 positions: fits
    gk.gk_sync(gkctx)
    got = ids4.cpu().numpy()
    assert np.array_equal(got[:, :Tp], prompt.reshape(B, Tp))
    assert ((got[:, Tp:] >= 0) & (got[:, Tp:] < s.V)).all()
    kv.close()


def _launches_per_step(gkctx, s, B, n_steps=4, Tp=6):
    import torch

    from gpt_decoder_gb300 import gk

    prompt, params, m, kv = _setup(gkctx, s, B, Tp, 9, Tp + n_steps)
    logits = torch.empty(B, s.V, device="cuda")
    tok = torch.as_tensor(prompt[:, -1].copy()).cuda()
    gk.gk_prefill(gkctx, m.params, kv, torch.as_tensor(prompt.reshape(-1)).cuda(), Tp, logits)
    l0 = gk.gk_launch_count(gkctx)
    for _ in range(n_steps):
        gk.gk_decode_step(gkctx, m.params, kv, tok, logits, tok, None)
    gk.gk_sync(gkctx)
    kv.close()
    return (gk.gk_launch_count(gkctx) - l0) / n_steps


def test_decode_step_is_one_persistent_launch_plus_selection(gkctx):
    """A decode step of a model narrower than 512 at batch 1 or 2 runs as one persistent kernel
    (embedding, every layer, ln_f and the head), then the selection and the position advance:
    three launches. From batch 4 on, and for models of width 512 and more (GPT-2-124M is 768),
    the step keeps the per-layer launches (five per layer)."""
    s = synth.GptShape(V=64, T=32, C=96, H=4, L=4)
    assert _launches_per_step(gkctx, s, 1) == 3
    assert _launches_per_step(gkctx, s, 2) == 3
    assert _launches_per_step(gkctx, s, 4) > 5 * s.L
    wide = synth.GptShape(V=64, T=32, C=512, H=8, L=2)
    assert _launches_per_step(gkctx, wide, 1) > 5 * wide.L


@pytest.mark.parametrize("B", [1, 3])
def test_deep_model_decodes_with_per_layer_launches(gkctx, B):
    """A model deeper than the persistent kernel's parameters hold (25 layers) decodes with the
    per-layer launches (five per layer), against the oracle teacher-forced."""
    s = synth.GptShape(V=64, T=32, C=32, H=2, L=25)
    assert _launches_per_step(gkctx, s, B) > 5 * 25
    err, mism, near, _, _ = _teacher_forced(gkctx, s, B, 8, 12, 4)
    assert err <= 5e-4
    assert mism == near, (mism, near)
