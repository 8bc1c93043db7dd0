"""libgk's safetensors reader and writer (host code, no GPU) against the oracle's: files written
by either are read by the other, the two writers produce the same bytes, and malformed files are
refused with the documented status."""
import os
import struct

import numpy as np
import pytest

import synth
from oracle import safetensors as ost


@pytest.fixture(scope="module")
def gk():
    from gpt_decoder_gb300 import gk as lib

    return lib


def _items(seed=3):
    st = synth.Stream(seed)
    return [("wte.weight", st.normal(64 * 12).reshape(64, 12)), ("h.0.ln_1.bias", st.normal(12)),
            ("scalar", np.array(-1.5, np.float32)), ("empty", np.zeros((0, 4), np.float32)),
            ('quote"back\\slash/é', st.normal(6).reshape(1, 2, 3))]


def test_writers_agree_byte_for_byte(gk, tmp_path):
    a, b = tmp_path / "ours.safetensors", tmp_path / "oracle.safetensors"
    gk.write_safetensors(a, _items(), {"format": "pt", "step": "7"})
    ost.write(b, _items(), {"format": "pt", "step": "7"})
    assert a.read_bytes() == b.read_bytes()
    assert not os.path.exists(str(a) + ".tmp")


def test_reads_what_the_oracle_writes(gk, tmp_path):
    p = tmp_path / "o.safetensors"
    ost.write(p, _items(), {"k": "v"})
    with gk.SafeTensors(p) as f:
        assert f.names() == [k for k, _ in _items()]
        assert f.metadata("k") == "v" and f.metadata("missing") is None
        for k, v in _items():
            assert f.shape(k) == v.shape and f.dtype(k) == "F32"
            np.testing.assert_array_equal(f.read(k), v)


def test_oracle_reads_what_we_write(gk, tmp_path):
    p = tmp_path / "g.safetensors"
    gk.write_safetensors(p, _items())
    meta, got = ost.read(p)
    assert meta == {} and list(got) == [k for k, _ in _items()]
    for k, v in _items():
        assert got[k].shape == v.shape
        np.testing.assert_array_equal(got[k], v)


def test_pages_gpt2_header_entry(gk, tmp_path, page):
    """The pages' printed GPT-2 header entry (h.3.ln_2.bias, F32, [768], data_offsets
    [202420224, 202423296]) in a sparse file: the reader finds the 768 numbers at 8 + N + begin."""
    begin, end = int(page["safetensors.gpt2.ln_2_bias.begin"]), int(page["safetensors.gpt2.ln_2_bias.end"])
    text = ('{"__metadata__":{"format":"pt"},"h.3.ln_2.bias":{"dtype":"F32","shape":[768],'
            f'"data_offsets":[{begin},{end}]}}}}').encode()
    vals = np.linspace(-1, 1, 768, dtype=np.float32)
    p = tmp_path / "gpt2_fragment.safetensors"
    with open(p, "wb") as f:
        f.write(struct.pack("<Q", len(text)) + text)
        f.seek(8 + len(text) + begin)
        f.write(vals.tobytes())
    with gk.SafeTensors(p) as f:
        assert f.names() == ["h.3.ln_2.bias"] and f.metadata("format") == "pt"
        np.testing.assert_array_equal(f.read("h.3.ln_2.bias"), vals)


def _raw(p, text, data=b""):
    p.write_bytes(struct.pack("<Q", len(text)) + text + data)
    return p


@pytest.mark.parametrize("text,data,at_open", [
    (b'{"x":{"dtype":"F32","shape":[2],"data_offsets":[0,8]', b"\0" * 8, True),      # unterminated JSON
    (b'{"x":{"dtype":"F32","shape":[2],"data_offsets":[0,8]},"x":{"dtype":"F32","shape":[0],'
     b'"data_offsets":[8,8]}}', b"\0" * 8, True),                                      # duplicate name
    (b'{"x":{"dtype":"F32","shape":[4],"data_offsets":[0,16]}}', b"\0" * 8, True),    # past the end
    (b'{"x":{"dtype":"F32","shape":[-1],"data_offsets":[0,0]}}', b"", True),           # negative extent
    (b'{"x":{"shape":[1],"data_offsets":[0,4]}}', b"\0" * 4, True),                    # no dtype
    (b'{"__metadata__":{"a":1}}', b"", True),                                           # non-string metadata
    (b'[1,2]', b"", True),                                                              # not an object
    (b'{"\xc3(":{"dtype":"F32","shape":[0],"data_offsets":[0,0]}}', b"", True),      # invalid UTF-8
    (b'{"\\ud800x":{"dtype":"F32","shape":[0],"data_offsets":[0,0]}}', b"", True),  # lone surrogate
    (b'{"\\udc00":{"dtype":"F32","shape":[0],"data_offsets":[0,0]}}', b"", True),   # lone low surrogate
    (b'{"x":{"dtype":"F16","shape":[2],"data_offsets":[0,4]}}', b"\0" * 4, False),    # dtype refused
    (b'{"x":{"dtype":"F32","shape":[3],"data_offsets":[0,8]}}', b"\0" * 8, False),    # offsets vs shape
    (b'{"x":{"dtype":"F32","shape":[4294967296,4294967296],"data_offsets":[0,0]}}', b"", True),  # count wraps
    (b'{"x":{"dtype":"F32","shape":[4611686018427387904,4],"data_offsets":[0,0]}}', b"", True),  # bytes wrap
])
def test_malformed_files_are_refused(gk, tmp_path, text, data, at_open):
    p = _raw(tmp_path / "bad.safetensors", text, data)
    if at_open:
        with pytest.raises(gk.GkError) as e:
            gk.SafeTensors(p)
        assert e.value.status == gk.GK_ERR_FORMAT
        return
    with gk.SafeTensors(p) as f:
        with pytest.raises(gk.GkError) as e:
            f.read("x")
        assert e.value.status == gk.GK_ERR_FORMAT
        assert "F16" in str(e.value) or "offsets" in str(e.value)


def test_io_and_argument_errors(gk, tmp_path):
    with pytest.raises(gk.GkError) as e:
        gk.SafeTensors(tmp_path / "missing.safetensors")
    assert e.value.status == gk.GK_ERR_IO
    p = _raw(tmp_path / "short.safetensors", b"", b"")
    p.write_bytes(b"\1\0")
    with pytest.raises(gk.GkError) as e:
        gk.SafeTensors(p)
    assert e.value.status == gk.GK_ERR_FORMAT
    with pytest.raises(gk.GkError) as e:
        gk.write_safetensors(tmp_path / "dup.safetensors", [("a", np.zeros(1, np.float32))] * 2)
    assert e.value.status == gk.GK_ERR_ARG
    assert not os.path.exists(tmp_path / "dup.safetensors")
    q = tmp_path / "ok.safetensors"
    gk.write_safetensors(q, [("a", np.zeros(3, np.float32))])
    import torch

    with gk.SafeTensors(q) as f:
        with pytest.raises(gk.GkError) as e:
            f.read("a", out=torch.zeros(4))  # size differs from the tensor's
        assert e.value.status == gk.GK_ERR_ARG
        with pytest.raises(KeyError):
            f.read("b")


def test_json_escapes_round_trip(gk, tmp_path):
    p = tmp_path / "esc.safetensors"
    text = '{"tab\\there\\u00e9\\/":{"dtype":"F32","shape":[1],"data_offsets":[0,4]}}'.encode()
    _raw(p, text, np.float32(2.5).tobytes())
    with gk.SafeTensors(p) as f:
        assert f.names() == ["tab\thereé/"]
        assert f.read("tab\thereé/")[0] == 2.5
    # a surrogate pair is one character outside the basic plane
    _raw(p, '{"\\ud83d\\ude00":{"dtype":"F32","shape":[0],"data_offsets":[0,0]}}'.encode())
    with gk.SafeTensors(p) as f:
        assert f.names() == ["\U0001F600"]


def test_mutated_headers_are_opened_or_refused(gk, tmp_path):
    """Byte flips, insertions and truncations of a valid file's header either still parse or
    are refused with GK_ERR_FORMAT; the parser never reads past what the file holds."""
    import random

    p = tmp_path / "base.safetensors"
    ost.write(p, _items(), {"format": "pt"})
    base = p.read_bytes()
    (n,) = struct.unpack("<Q", base[:8])
    rng = random.Random(1)
    alphabet = b'{}[]:,"\\0123456789-eE.tfnu ' + bytes(range(0x7F, 0x83)) + b"\xc3\xa9\xff"
    q = tmp_path / "mut.safetensors"
    outcomes = set()
    for trial in range(400):
        hdr = bytearray(base[8:8 + n])
        for _ in range(rng.randint(1, 4)):
            kind, at = rng.randrange(3), rng.randrange(len(hdr))
            if kind == 0:
                hdr[at] = rng.choice(alphabet)
            elif kind == 1:
                hdr[at:at] = bytes([rng.choice(alphabet)])
            else:
                del hdr[at:]
                break
        q.write_bytes(struct.pack("<Q", len(hdr)) + bytes(hdr) + base[8 + n:])
        try:
            with gk.SafeTensors(q) as f:
                for name in f.names():
                    try:
                        f.read(name)
                    except gk.GkError as e:  # an entry whose offsets no longer match its shape
                        assert "GK_ERR_FORMAT" in str(e), str(e)
            outcomes.add("ok")
        except gk.GkError as e:
            assert "GK_ERR_FORMAT" in str(e), str(e)
            outcomes.add("refused")
    assert outcomes == {"ok", "refused"}


def test_checkpoint_order_is_gpt2s():
    from gpt_decoder_gb300.checkpoint import _gpt2_order

    names = [k for k, _ in synth.param_names_shapes(synth.TINY)]
    scrambled = {k: i for i, k in enumerate(["wte.weight", "wpe.weight", "ln_f.weight", "ln_f.bias"]
                                             + [k for k in names if k.startswith("h.")])}
    assert [k for k, _ in _gpt2_order(scrambled)] == names
