"""Oracle reader and writer of the safetensors file format, float32 tensors.

TEST INFRASTRUCTURE ONLY (see the package docstring): never imported by the product path.

[LM4] "Build a language model in C# from scratch (4): running GPT-2 weights", "The safetensors
format": the first 8 bytes hold the header length N as a little-endian unsigned 64-bit
integer; the next N bytes are a JSON object mapping each tensor name to its dtype, shape and
data_offsets [begin, end) (byte offsets relative to the end of the header), plus an optional
"__metadata__" entry that is not a tensor; the rest of the file is the tensors' raw bytes.
Only F32 is read; any other dtype is refused.

Readings where the pages are silent: the writer lays the tensors out back to back in the
order given, pads the JSON with spaces to a multiple of 8 bytes (so the data starts aligned;
JSON allows the trailing whitespace), keeps non-ASCII names as UTF-8 rather than JSON
unicode escapes, and stores float32 little-endian.
"""
from __future__ import annotations

import json
import math
import struct

import numpy as np


class FormatError(ValueError):
    pass


def write(path, tensors, metadata=None):
    """tensors: a sequence of (name, float32 array) or a dict; metadata: str -> str."""
    items = list(tensors.items()) if isinstance(tensors, dict) else list(tensors)
    header, begin = {}, 0
    if metadata:
        header["__metadata__"] = {str(k): str(v) for k, v in metadata.items()}
    for name, arr in items:
        a = np.asarray(arr)
        if a.dtype != np.float32:
            raise FormatError(f"{name}: only float32 is written")
        header[name] = {"dtype": "F32", "shape": list(a.shape), "data_offsets": [begin, begin + a.nbytes]}
        begin += a.nbytes
    text = json.dumps(header, separators=(",", ":"), ensure_ascii=False).encode("utf-8")
    text += b" " * (-len(text) % 8)
    with open(path, "wb") as f:
        f.write(struct.pack("<Q", len(text)))
        f.write(text)
        for _, arr in items:
            f.write(np.ascontiguousarray(arr, dtype="<f4").tobytes())


def read_header(path):
    """(header length N, the parsed JSON object) of a file."""
    with open(path, "rb") as f:
        raw = f.read(8)
        if len(raw) != 8:
            raise FormatError("shorter than the 8-byte header length")
        (n,) = struct.unpack("<Q", raw)
        text = f.read(n)
        if len(text) != n:
            raise FormatError("header runs past the end of the file")
    try:
        obj = json.loads(text.decode("utf-8"))  # JSON text is UTF-8
    except (UnicodeDecodeError, json.JSONDecodeError) as e:
        raise FormatError(f"header: {e}") from None
    if not isinstance(obj, dict):
        raise FormatError("header is not a JSON object")
    return n, obj


def read(path):
    """(metadata dict, {name: float32 array}) of every tensor, in header order."""
    n, obj = read_header(path)
    meta = obj.get("__metadata__", {})
    data_start = 8 + n
    out = {}
    with open(path, "rb") as f:
        f.seek(0, 2)
        size = f.tell()
        for name, e in obj.items():
            if name == "__metadata__":
                continue
            if e["dtype"] != "F32":
                raise FormatError(f"{name}: dtype {e['dtype']}, only F32 is handled")
            begin, end = e["data_offsets"]
            shape = tuple(int(s) for s in e["shape"])
            count = math.prod(shape)  # exact (Python integers): a shape whose size overflows is refused below
            if end - begin != 4 * count or begin < 0 or data_start + end > size:
                raise FormatError(f"{name}: data_offsets {begin}, {end} do not fit shape {shape} and the file")
            f.seek(data_start + begin)
            out[name] = np.frombuffer(f.read(end - begin), dtype="<f4").reshape(shape).astype(np.float32)
    return meta, out
