"""Plain GGUF reader (test infrastructure): the oracle of the library's
container parser.

It follows the file structure of "12 -- llama.cpp / GGUF / Local Inference
Mastery", "Part 1 -- The GGUF format (bit-level)", field by field in the
order the figure lists them:
  header        magic "GGUF" (4 bytes), version uint32, tensor_count uint64,
                metadata_kv_count uint64;
  metadata      per entry: key (length-prefixed string), value type, value;
  tensor infos  per tensor: name, n_dims, shape, type, offset;
  padding       to the alignment ("typically 32 bytes");
  tensor data   at the offsets, counted from the start of the data section.
Little-endian.  Not on the page, taken from the GGUF specification it cites:
string lengths are uint64 (versions 2 and 3), value types are uint32 codes
0 u8, 1 i8, 2 u16, 3 i16, 4 u32, 5 i32, 6 f32, 7 bool, 8 string, 9 array
(uint32 element type, uint64 count, elements), 10 u64, 11 i64, 12 f64, and a
"general.alignment" uint32 entry overrides the 32-byte default.

Only the tests may import this module.  Errors raise ValueError.
"""
from __future__ import annotations

import struct

_SCALAR = {0: "<B", 1: "<b", 2: "<H", 3: "<h", 4: "<I", 5: "<i", 6: "<f", 7: "<?", 10: "<Q", 11: "<q", 12: "<d"}
_STRING, _ARRAY = 8, 9


class _Buf:
    def __init__(self, data: bytes):
        self.data, self.pos = data, 0

    def take(self, n: int) -> bytes:
        if n < 0 or self.pos + n > len(self.data):
            raise ValueError("truncated")
        b = self.data[self.pos:self.pos + n]
        self.pos += n
        return b

    def unpack(self, fmt: str):
        return struct.unpack(fmt, self.take(struct.calcsize(fmt)))[0]

    def string(self) -> bytes:
        return self.take(self.unpack("<Q"))


def _value(buf: _Buf, vtype: int, depth: int = 0):
    if vtype in _SCALAR:
        return buf.unpack(_SCALAR[vtype])
    if vtype == _STRING:
        return buf.string()
    if vtype == _ARRAY and depth < 8:
        etype = buf.unpack("<I")
        n = buf.unpack("<Q")
        return (etype, [_value(buf, etype, depth + 1) for _ in range(n)])
    raise ValueError(f"bad value type {vtype}")


def read(data: bytes) -> dict:
    """Parse a GGUF image: {'version', 'kv': {key: (type, value)}, 'tensors':
    [(name, dims, ggml_type, offset)], 'alignment', 'data_offset'}.  Strings
    are returned as bytes; arrays as (element type, [values])."""
    buf = _Buf(data)
    if buf.take(4) != b"GGUF":
        raise ValueError("magic")
    version = buf.unpack("<I")
    if version not in (2, 3):
        raise ValueError("version")
    n_tensors = buf.unpack("<Q")
    n_kv = buf.unpack("<Q")
    kv = {}
    for _ in range(n_kv):
        key = buf.string().decode("utf-8", "surrogateescape")
        vtype = buf.unpack("<I")
        kv[key] = (vtype, _value(buf, vtype))
    alignment = 32
    if "general.alignment" in kv:
        vtype, a = kv["general.alignment"]
        if vtype != 4 or a <= 0 or a & (a - 1):
            raise ValueError("alignment")
        alignment = a
    tensors = []
    for _ in range(n_tensors):
        name = buf.string().decode("utf-8", "surrogateescape")
        n_dims = buf.unpack("<I")
        dims = [buf.unpack("<Q") for _ in range(n_dims)]
        gtype = buf.unpack("<I")
        offset = buf.unpack("<Q")
        tensors.append((name, dims, gtype, offset))
    data_offset = (buf.pos + alignment - 1) // alignment * alignment
    return {"version": version, "kv": kv, "tensors": tensors, "alignment": alignment, "data_offset": data_offset}
