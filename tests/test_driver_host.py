"""Host-side checks of the training-step driver: buffer plan and parameter views (no GPU)."""
import numpy as np
import pytest

import synth


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_driver_buffers_and_views(mode):
    torch = pytest.importorskip("torch")
    from gpt_decoder_gb300 import gk
    from gpt_decoder_gb300.model import Gpt

    s = synth.GptShape(V=50, T=8, C=16, H=2, L=3)
    m = Gpt(None, s.V, s.T, s.C, s.H, s.L, 2, mode=mode, device="cpu")
    assert m.ldt == [gk.GK_F32 if mode == "fp32" else gk.GK_BF16] * 3
    assert m.split == ([False] * 3 if mode == "fp32" else [True, True, False])
    cuts = m.adamw_cuts()
    assert cuts[0][0] == 0 and cuts[-1][1] == m.numel
    assert all(a[1] == b[0] for a, b in zip(cuts, cuts[1:]))
    assert all(d == (e <= m.n_decay) for (_, e, d, _) in cuts)
    if mode == "bf16":
        lo_spans = [c for c in cuts if c[3]]
        assert lo_spans == [(m.hi_lo, m.hi_hi, 1, True)]
        assert m.hi_hi - m.hi_lo == 2 * 12 * s.C * s.C == m.params_bf16_lo.numel()
    assert m.Vp % 64 == 0 and m.Vp >= s.V
    views = m.named_slices(m.params)
    assert set(views) == {n for n, _ in synth.param_names_shapes(s)}
    for name, shape in synth.param_names_shapes(s):
        assert tuple(views[name].shape) == shape
    # every element of the flat buffer belongs to exactly one view
    cover = torch.zeros(m.numel, dtype=torch.int32)
    marks = m.named_slices(cover)
    for v in marks.values():
        v += 1
    assert int(cover.min()) == 1 and int(cover.max()) == 1
    _, _, params = synth.training_case(s, 2, 0)
    for k, v in params.items():
        views[k].copy_(torch.as_tensor(v))
        np.testing.assert_array_equal(views[k].numpy(), v)
