"""Checkpoints of a Gpt as safetensors files ([LM4] "The safetensors format", written and read
by libgk's gk_st_* functions): the parameters under their GPT-2 names ("wte.weight",
"h.0.attn.c_attn.weight", ...; a file holding only these loads like the pages' GPT-2 file),
the AdamW moments as "adamw.m.<name>" and "adamw.v.<name>", and the optimizer's step count in
the metadata. The tensors move between the file and the device buffers directly (staged
through host memory by the library)."""
from __future__ import annotations

from . import gk

FORMAT = "gpt_decoder_gb300"


def _gpt2_order(named):
    """(name, view) pairs in GPT-2's order: embeddings, the blocks in order, then ln_f."""
    keys = list(named)
    order = ([k for k in keys if not k.startswith(("h.", "ln_f."))] + [k for k in keys if k.startswith("h.")]
             + [k for k in keys if k.startswith("ln_f.")])
    return [(k, named[k]) for k in order]


def save(path, model, with_optimizer=True):
    """Write `model`'s parameters (and, with_optimizer, its AdamW state) to `path`."""
    import torch

    torch.cuda.current_stream().synchronize()
    gk.gk_sync(model.ctx)
    tensors = _gpt2_order(model.named_slices(model.params))
    if with_optimizer:
        tensors += [("adamw.m." + k, v) for k, v in _gpt2_order(model.named_slices(model.m))]
        tensors += [("adamw.v." + k, v) for k, v in _gpt2_order(model.named_slices(model.v))]
    meta = {"format": FORMAT, "step": str(model.step_count),
            "shape": f"V={model.V} T={model.T} C={model.C} H={model.H} L={model.L}"}
    gk.write_safetensors(path, [(k, v.contiguous()) for k, v in tensors], meta)


def load(path, model):
    """Read parameters (and the AdamW state and step count, when the file has them) into
    `model`; every parameter tensor of the model must be in the file with its shape."""
    import torch

    torch.cuda.current_stream().synchronize()
    with gk.SafeTensors(path) as f:
        names = set(f.names())
        groups = [("", model.params)]
        if "adamw.m.wte.weight" in names:
            groups += [("adamw.m.", model.m), ("adamw.v.", model.v)]
        for prefix, buf in groups:
            for k, view in model.named_slices(buf).items():
                if f.shape(prefix + k) != tuple(view.shape):
                    raise ValueError(f"{prefix + k}: shape {f.shape(prefix + k)} in the file, {tuple(view.shape)} here")
                f.read(prefix + k, out=view)
        step = f.metadata("step")
        if len(groups) > 1 and step is not None:
            model.step_count = int(step)
    model.refresh_bf16()
