"""Pins of the oracle's safetensors reader and writer ([LM4] "The safetensors format"): the byte
layout checked by hand, the pages' printed GPT-2 header entry read from a file laid out as
the pages describe, the GPT-2 tensor table, round trips and refusals."""
import json
import struct

import numpy as np
import pytest

import synth
from oracle import safetensors as ost


def test_byte_layout_by_hand(tmp_path):
    a = np.arange(6, dtype=np.float32).reshape(2, 3) - 2.5
    b = np.array([1e-30, -7.25], np.float32)
    p = tmp_path / "t.safetensors"
    ost.write(p, [("a", a), ("b", b)], {"format": "pt"})
    raw = p.read_bytes()
    (n,) = struct.unpack("<Q", raw[:8])
    assert n % 8 == 0
    hdr = json.loads(raw[8:8 + n])
    assert hdr["__metadata__"] == {"format": "pt"}
    assert hdr["a"] == {"dtype": "F32", "shape": [2, 3], "data_offsets": [0, 24]}
    assert hdr["b"] == {"dtype": "F32", "shape": [2], "data_offsets": [24, 32]}
    data = raw[8 + n:]
    assert data == a.astype("<f4").tobytes() + b.astype("<f4").tobytes()


def test_pages_gpt2_header_entry(tmp_path, page):
    """The pages' loader prints the start of GPT-2's header, {"__metadata__":{"format":"pt"},
    "h.3.ln_2.bias":{"dtype":"F32","shape":[768],"data_offsets":[202420224,202423296]}, ...:
    a file with that entry (data written at 8 + N + begin, the rest of the file sparse) reads
    back those 768 numbers, so the offsets count from the end of the header and the metadata
    entry is skipped."""
    begin, end = int(page["safetensors.gpt2.ln_2_bias.begin"]), int(page["safetensors.gpt2.ln_2_bias.end"])
    text = ('{"__metadata__":{"format":"pt"},"h.3.ln_2.bias":{"dtype":"F32","shape":[768],'
            f'"data_offsets":[{begin},{end}]}}}}').encode()
    vals = np.linspace(-1, 1, 768, dtype=np.float32)
    p = tmp_path / "gpt2_fragment.safetensors"
    with open(p, "wb") as f:
        f.write(struct.pack("<Q", len(text)) + text)
        f.seek(8 + len(text) + begin)
        f.write(vals.tobytes())
    assert end - begin == 4 * 768
    meta, t = ost.read(p)
    assert meta == {"format": "pt"} and list(t) == ["h.3.ln_2.bias"]
    np.testing.assert_array_equal(t["h.3.ln_2.bias"], vals)


def test_gpt2_tensor_table(page):
    # 148 parameters, 124,439,808 numbers; the shapes the pages' loader prints
    names = dict(synth.param_names_shapes(synth.GPT2_124M))
    assert len(names) == int(page["safetensors.gpt2.params"])
    assert sum(int(np.prod(s)) for s in names.values()) == int(page["safetensors.gpt2.numbers"])
    assert names["wte.weight"] == (50257, 768) and names["wpe.weight"] == (1024, 768)
    assert names["h.0.attn.c_attn.weight"] == (768, 2304) and names["h.0.attn.c_proj.weight"] == (768, 768)
    assert names["h.0.mlp.c_fc.weight"] == (768, 3072) and names["h.0.mlp.c_proj.weight"] == (3072, 768)
    assert names["h.3.ln_2.bias"] == (768,) and names["ln_f.weight"] == (768,)


def test_round_trip_shapes(tmp_path):
    st = synth.Stream(9)
    items = [("scalar", np.array(3.5, np.float32)), ("empty", np.zeros((0,), np.float32)),
             ("m", st.normal(35).reshape(5, 7)), ("t3", st.normal(24).reshape(2, 3, 4))]
    p = tmp_path / "r.safetensors"
    ost.write(p, items)
    meta, got = ost.read(p)
    assert meta == {} and list(got) == [k for k, _ in items]
    for k, v in items:
        assert got[k].shape == v.shape
        np.testing.assert_array_equal(got[k], v)


def test_refusals(tmp_path):
    p = tmp_path / "f16.safetensors"
    text = b'{"x":{"dtype":"F16","shape":[2],"data_offsets":[0,4]}}'
    p.write_bytes(struct.pack("<Q", len(text)) + text + b"\0" * 4)
    with pytest.raises(ost.FormatError, match="only F32"):
        ost.read(p)
    q = tmp_path / "short.safetensors"
    text = b'{"x":{"dtype":"F32","shape":[4],"data_offsets":[0,16]}}'
    q.write_bytes(struct.pack("<Q", len(text)) + text + b"\0" * 8)  # 8 of 16 bytes
    with pytest.raises(ost.FormatError):
        ost.read(q)
    u = tmp_path / "utf8.safetensors"
    text = b'{"\xc3(":{"dtype":"F32","shape":[0],"data_offsets":[0,0]}}'
    u.write_bytes(struct.pack("<Q", len(text)) + text)
    with pytest.raises(ost.FormatError):
        ost.read(u)
    r = tmp_path / "trunc.safetensors"
    r.write_bytes(struct.pack("<Q", 100) + b"{}")
    with pytest.raises(ost.FormatError):
        ost.read(r)


def test_shape_whose_size_overflows_is_refused(tmp_path):
    # 2^32 x 2^32 elements: a 64-bit product wraps to 0 and would match empty data_offsets
    p = tmp_path / "wrap.safetensors"
    text = b'{"x":{"dtype":"F32","shape":[4294967296,4294967296],"data_offsets":[0,0]}}'
    p.write_bytes(struct.pack("<Q", len(text)) + text)
    with pytest.raises(ost.FormatError):
        ost.read(p)
