"""A minimal GGUF (version 3) file writer for the reader's tests.

Test infrastructure: it writes the published container layout (little-endian
header "GGUF", u32 version, u64 tensor count, u64 key-value count; the
key-value pairs; the tensor infos; padding to the alignment; the tensor data,
each tensor at an aligned offset from the data start) with numpy and struct,
and shares no code with the library's reader.  GGUF Support Proposal for
mobius, 1.1 "Overview": metadata key-value pairs plus tensors with a
per-tensor type.  Tensor dims are written contiguous-first: a weight W[N, K]
gets dims (K, N)."""
from __future__ import annotations

import struct

import numpy as np

U8, I8, U16, I16, U32, I32, F32, BOOL, STRING, ARRAY, U64, I64, F64 = range(13)
_SCALAR = {U8: "<B", I8: "<b", U16: "<H", I16: "<h", U32: "<I", I32: "<i", F32: "<f", BOOL: "<?", U64: "<Q",
           I64: "<q", F64: "<d"}


def _string(s) -> bytes:
    b = s.encode("utf-8") if isinstance(s, str) else bytes(s)
    return struct.pack("<Q", len(b)) + b


def _value(vtype, v) -> bytes:
    if vtype == STRING:
        return _string(v)
    if vtype == ARRAY:
        etype, items = v
        out = struct.pack("<IQ", etype, len(items))
        return out + b"".join(_value(etype, x) for x in items)
    return struct.pack(_SCALAR[vtype], v)


def gguf_bytes(kv, tensors, alignment=None, version=3) -> bytes:
    """kv: [(key, value type, value)] (an array value is (element type, items));
    tensors: [(name, ggml type id, dims contiguous-first, raw bytes)].
    With alignment given, a general.alignment u32 pair is appended to kv."""
    kv = list(kv)
    align = 32
    if alignment is not None:
        kv.append(("general.alignment", U32, alignment))
        align = alignment
    head = b"GGUF" + struct.pack("<IQQ", version, len(tensors), len(kv))
    for key, vt, v in kv:
        head += _string(key) + struct.pack("<I", vt) + _value(vt, v)
    offsets, off = [], 0
    for _, _, _, raw in tensors:
        offsets.append(off)
        off += -(-len(raw) // align) * align
    for (name, ttype, dims, _), o in zip(tensors, offsets):
        head += _string(name) + struct.pack("<I", len(dims)) + b"".join(struct.pack("<Q", d) for d in dims)
        head += struct.pack("<IQ", ttype, o)
    data_start = -(-len(head) // align) * align
    out = bytearray(head + b"\0" * (data_start - len(head)))
    for i, ((_, _, _, raw), o) in enumerate(zip(tensors, offsets)):
        assert len(out) == data_start + o
        out += bytes(raw)
        if i + 1 < len(tensors):           # padding between tensors, none after the last
            out += b"\0" * (-(-len(raw) // align) * align - len(raw))
    return bytes(out)


def write(path, kv, tensors, alignment=None, version=3):
    data = gguf_bytes(kv, tensors, alignment, version)
    with open(path, "wb") as f:
        f.write(data)
    return data


def weight_tensor(name, qtype, blocks: np.ndarray, N, K):
    """A block-quantized weight W[N, K] stored as GGUF does: dims (K, N)."""
    return (name, qtype, (K, N), np.ascontiguousarray(blocks).tobytes())
