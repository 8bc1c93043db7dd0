"""Checkpoints through libgk's safetensors code: device tensors written and read back
bit-exactly, a saved model read by the oracle's reader under the GPT-2 names, and training resumed
from a checkpoint giving the same losses as training that never stopped."""
import numpy as np
import pytest

import synth
from oracle import safetensors as ost

pytestmark = pytest.mark.gpu


def test_device_tensors_round_trip(gkctx, tmp_path):
    import torch

    from gpt_decoder_gb300 import gk

    st = synth.Stream(4)
    big = torch.as_tensor(st.normal((1 << 24) + 5)).cuda()  # larger than the 64 MB staging chunk
    small = torch.as_tensor(st.normal(12).reshape(3, 4)).cuda()
    p = tmp_path / "dev.safetensors"
    gk.write_safetensors(p, [("big", big), ("small", small)], {"note": "device"})
    meta, host = ost.read(p)
    assert meta == {"note": "device"}
    np.testing.assert_array_equal(host["big"], big.cpu().numpy())
    out_big, out_small = torch.empty_like(big), torch.empty_like(small)
    with gk.SafeTensors(p) as f:
        f.read("big", out=out_big)
        f.read("small", out=out_small)
    assert torch.equal(out_big, big) and torch.equal(out_small, small)


@pytest.mark.parametrize("mode", ["fp32", "bf16"])
def test_resume_from_checkpoint_matches_uninterrupted_training(gkctx, tmp_path, mode):
    import torch

    from gpt_decoder_gb300 import checkpoint, gk
    from gpt_decoder_gb300.model import Gpt

    s = synth.TINY
    ids, targets, params = synth.training_case(s, 4, 11)
    d_ids = torch.as_tensor(ids.reshape(-1)).cuda()
    d_tg = torch.as_tensor(targets.reshape(-1)).cuda()
    a = Gpt(gkctx, s.V, s.T, s.C, s.H, s.L, 4, mode=mode)
    a.load(params)
    for _ in range(3):
        a.train_step(d_ids, d_tg, 1e-3, 0.01)
    path = tmp_path / "ckpt.safetensors"
    checkpoint.save(path, a)
    straight = [a.train_step(d_ids, d_tg, 1e-3, 0.01).item() for _ in range(3)]

    b = Gpt(gkctx, s.V, s.T, s.C, s.H, s.L, 4, mode=mode)
    checkpoint.load(path, b)
    assert b.step_count == 3
    resumed = [b.train_step(d_ids, d_tg, 1e-3, 0.01).item() for _ in range(3)]
    gk.gk_sync(gkctx)
    assert resumed == straight
    assert torch.equal(a.params, b.params) and torch.equal(a.m, b.m) and torch.equal(a.v, b.v)

    # the file holds every GPT-2 parameter under its name, readable by the oracle's reader
    meta, host = ost.read(path)
    names = [k for k, _ in synth.param_names_shapes(s)]
    assert [k for k in host if not k.startswith("adamw.")] == names
    assert meta["format"] == "gpt_decoder_gb300" and meta["step"] == "3"
    for k, shape in synth.param_names_shapes(s):
        assert host[k].shape == shape


def test_weights_only_file_loads_like_a_gpt2_checkpoint(gkctx, tmp_path):
    """A file with only the GPT-2 parameter names (as the pages' GPT-2 file has) loads the
    weights and leaves the optimizer state alone."""
    import torch

    from gpt_decoder_gb300 import checkpoint
    from gpt_decoder_gb300.model import Gpt

    s = synth.TINY
    _, _, params = synth.training_case(s, 2, 12)
    p = tmp_path / "weights.safetensors"
    ost.write(p, [(k, params[k]) for k, _ in synth.param_names_shapes(s)], {"format": "pt"})
    m = Gpt(gkctx, s.V, s.T, s.C, s.H, s.L, 2, mode="fp32")
    checkpoint.load(p, m)
    views = m.named_slices(m.params)
    for k, _ in synth.param_names_shapes(s):
        np.testing.assert_array_equal(views[k].cpu().numpy(), params[k])
    assert m.step_count == 0 and not torch.any(m.m)
