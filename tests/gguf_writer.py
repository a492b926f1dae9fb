"""Writes GGUF images for the tests (version 3 unless asked otherwise).

Layout from "12 -- llama.cpp / GGUF / Local Inference Mastery", "Part 1 -- The
GGUF format (bit-level)": header (magic "GGUF", uint32 version, uint64
tensor_count, uint64 metadata_kv_count), metadata entries (uint64-length key,
uint32 value type, value), tensor infos (name, uint32 n_dims, uint64 dims
innermost first, uint32 ggml type, uint64 offset from the data section),
padding to the alignment, tensor data.  Little-endian.  Value-type and ggml
type numbers are the GGUF specification's, which the page cites.
"""
from __future__ import annotations

import struct

VT = {"u8": 0, "i8": 1, "u16": 2, "i16": 3, "u32": 4, "i32": 5, "f32": 6, "bool": 7, "str": 8, "arr": 9,
      "u64": 10, "i64": 11, "f64": 12}
FMT = {"u8": "<B", "i8": "<b", "u16": "<H", "i16": "<h", "u32": "<I", "i32": "<i", "f32": "<f", "bool": "<?",
       "u64": "<Q", "i64": "<q", "f64": "<d"}
GGML = {"F32": 0, "F16": 1, "Q4_0": 2, "Q4_1": 3, "Q5_0": 6, "Q8_0": 8, "Q2_K": 10, "Q3_K": 11, "Q4_K": 12, "Q5_K": 13, "Q6_K": 14, "BF16": 30}


def _s(text: str | bytes) -> bytes:
    b = text.encode() if isinstance(text, str) else text
    return struct.pack("<Q", len(b)) + b


def _value(vtype, value) -> bytes:
    """vtype: a scalar name, 'str', or ('arr', element vtype)."""
    if isinstance(vtype, tuple):
        et = vtype[1]
        code = VT[et[0]] if isinstance(et, tuple) else VT[et]
        return struct.pack("<IQ", code, len(value)) + b"".join(_value(et, v) for v in value)
    if vtype == "str":
        return _s(value)
    return struct.pack(FMT[vtype], value)


def write(kvs, tensors, alignment: int | None = None, version: int = 3) -> bytes:
    """kvs: [(key, vtype, value)]; tensors: [(name, dims, ggml type name or
    number, data bytes)].  alignment: written as general.alignment when not
    None (and used for padding); 32 otherwise."""
    kvs = list(kvs)
    if alignment is not None:
        kvs.append(("general.alignment", "u32", alignment))
    align = alignment or 32
    out = bytearray(b"GGUF" + struct.pack("<IQQ", version, len(tensors), len(kvs)))
    for key, vtype, value in kvs:
        out += _s(key)
        code = VT["arr"] if isinstance(vtype, tuple) else VT[vtype]
        out += struct.pack("<I", code) + _value(vtype, value)
    offs, off = [], 0
    for name, dims, gt, data in tensors:
        offs.append(off)
        off = (off + len(data) + align - 1) // align * align
    for (name, dims, gt, data), o in zip(tensors, offs):
        code = GGML[gt] if isinstance(gt, str) else gt
        out += _s(name) + struct.pack("<I", len(dims)) + b"".join(struct.pack("<Q", d) for d in dims)
        out += struct.pack("<IQ", code, o)
    out += b"\0" * ((-len(out)) % align)
    # Each tensor is padded to the alignment, so tensor i starts at offs[i].
    for name, dims, gt, data in tensors:
        out += bytes(data)
        out += b"\0" * ((-len(bytes(data))) % align)
    return bytes(out)
