"""Writes small GGUF files for the reader's tests (test infrastructure).

Layout as "Go AI Inference: What is Inference?" draws it (section "GGUF: The
Whole Model in One File": header, typed key-value metadata, tensor
descriptors, data blob), with the field widths and type codes of GGUF
versions 2 and 3: little endian; magic GGUF, u32 version, u64 tensor count,
u64 metadata count; strings as u64 length + bytes; value types u8 0, i8 1,
u16 2, i16 3, u32 4, i32 5, f32 6, bool 7, string 8, array 9 (u32 element
type, u64 count, elements), u64 10, i64 11, f64 12; a descriptor is name,
u32 dim count, u64 dims (innermost first), u32 tensor type, u64 offset into
the blob; the blob starts at the first multiple of the alignment after the
descriptors and every tensor's offset is a multiple of it.
"""

from __future__ import annotations

import struct

TYPE = {"u8": 0, "i8": 1, "u16": 2, "i16": 3, "u32": 4, "i32": 5, "f32": 6, "bool": 7,
        "str": 8, "arr": 9, "u64": 10, "i64": 11, "f64": 12}
FMT = {"u8": "<B", "i8": "<b", "u16": "<H", "i16": "<h", "u32": "<I", "i32": "<i", "f32": "<f",
       "bool": "<B", "u64": "<Q", "i64": "<q", "f64": "<d"}


def _str(s: str) -> bytes:
    b = s.encode()
    return struct.pack("<Q", len(b)) + b


def _value(kind: str, v) -> bytes:
    if kind == "str":
        return _str(v)
    if kind == "arr":
        ekind, items = v
        out = struct.pack("<IQ", TYPE[ekind], len(items))
        return out + b"".join(_str(x) if ekind == "str" else struct.pack(FMT[ekind], x) for x in items)
    return struct.pack(FMT[kind], v)


def gguf_bytes(kvs, tensors, alignment: int = 32, version: int = 3) -> bytes:
    """kvs: [(key, kind, value)], arrays as ("arr", (element kind, [values]));
    tensors: [(name, type, dims innermost first, data bytes)]."""
    head = b"GGUF" + struct.pack("<IQQ", version, len(tensors), len(kvs))
    for key, kind, v in kvs:
        head += _str(key) + struct.pack("<I", TYPE[kind]) + _value(kind, v)
    offsets, off = [], 0
    for _, _, _, data in tensors:
        offsets.append(off)
        off += -(-len(data) // alignment) * alignment
    for (name, typ, dims, _), o in zip(tensors, offsets):
        head += _str(name) + struct.pack("<I", len(dims)) + b"".join(struct.pack("<Q", d) for d in dims)
        head += struct.pack("<IQ", typ, o)
    head += b"\0" * (-len(head) % alignment)
    blob = bytearray()
    for (_, _, _, data), o in zip(tensors, offsets):
        blob += b"\0" * (o - len(blob))
        blob += data
    return head + bytes(blob)


def write_gguf(path, kvs, tensors, alignment: int = 32, version: int = 3) -> None:
    with open(path, "wb") as f:
        f.write(gguf_bytes(kvs, tensors, alignment, version))
