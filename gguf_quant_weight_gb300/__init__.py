"""Python binding of libgguf_mm.so (matmul on GGUF block-quantized weights, GB300).

Argument marshalling only: every function has the name and the arguments of
the C entry point in include/gguf_mm.h.  Tensor arguments may be torch tensors
(their data_ptr() is passed) or raw integer device addresses; `stream` defaults
to torch's current CUDA stream.  A non-zero status raises GGUFError.  There is
no fallback: if the library is missing the import of a function fails loudly.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libgguf_mm.so")

# enums (same values as include/gguf_mm.h)
GGUF_Q4_0, GGUF_Q4_1, GGUF_Q5_0, GGUF_Q5_1 = 2, 3, 6, 7
GGUF_Q8_0, GGUF_Q4_K, GGUF_Q5_K, GGUF_Q6_K = 8, 12, 13, 14
GGUF_Q2_K, GGUF_Q3_K = 10, 11
GGUF_LAYOUT_BLOCKS, GGUF_LAYOUT_Q6K_PLANES = 0, 1
GGUF_DT_F32, GGUF_DT_F16, GGUF_DT_BF16 = 0, 1, 2
GGUF_PATH_AUTO, GGUF_PATH_GEMV, GGUF_PATH_FUSED = 0, 1, 2
GGUF_OP_GEMV, GGUF_OP_GEMM, GGUF_OP_ID, GGUF_OP_DENSE = 0, 1, 2, 3
GGUF_OK = 0
GGUF_ERR_INVALID_ARG, GGUF_ERR_UNSUPPORTED, GGUF_ERR_MISALIGNED = -1, -2, -3
GGUF_ERR_WORKSPACE, GGUF_ERR_CUDA, GGUF_ERR_TIMEOUT, GGUF_ERR_NO_DEVICE = -4, -5, -6, -7
GGUF_ERR_IO, GGUF_ERR_FORMAT, GGUF_ERR_NOT_FOUND = -8, -9, -10

BLOCK_VALUES = {GGUF_Q4_0: 32, GGUF_Q4_1: 32, GGUF_Q5_0: 32, GGUF_Q5_1: 32, GGUF_Q8_0: 32, GGUF_Q2_K: 256,
                GGUF_Q3_K: 256, GGUF_Q4_K: 256, GGUF_Q5_K: 256, GGUF_Q6_K: 256}
BLOCK_BYTES = {GGUF_Q4_0: 18, GGUF_Q4_1: 20, GGUF_Q5_0: 22, GGUF_Q5_1: 24, GGUF_Q8_0: 34, GGUF_Q2_K: 84,
               GGUF_Q3_K: 110, GGUF_Q4_K: 144, GGUF_Q5_K: 176, GGUF_Q6_K: 210}

_c_i64, _c_int, _c_sz, _c_vp = ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/gguf_mm.h
_SIGS = {
    "gguf_mm_workspace_size": (_c_sz, [_c_int, _c_int, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64]),
    "gguf_mm_gemv": (_c_int, [_c_vp, _c_int, _c_int, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_vp,
                              _c_int, _c_vp, _c_sz, _c_vp]),
    "gguf_mm_gemv_host": (_c_int, [_c_vp, _c_int, _c_int, _c_i64, _c_i64, _c_vp, _c_vp, _c_int, _c_i64, _c_vp,
                                   _c_vp, _c_vp, _c_vp, _c_int, _c_vp, _c_sz, _c_vp]),
    "gguf_mm_gemm": (_c_int, [_c_vp, _c_int, _c_int, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_vp,
                              _c_int, _c_vp, _c_sz, _c_int, _c_vp]),
    "gguf_mm_id": (_c_int, [_c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_i64,
                            _c_vp, _c_vp, _c_int, _c_vp, _c_sz, _c_vp]),
    "gguf_mm_id_slots": (_c_int, [_c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_i64,
                                  _c_vp, _c_vp, _c_int, _c_vp, _c_sz, _c_vp]),
    "gguf_mm_id_form": (_c_int, [_c_int, _c_i64, _c_i64]),
    "gguf_mm_id_path": (_c_int, [_c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_i64,
                                 _c_int, _c_vp, _c_vp, _c_int, _c_vp, _c_sz, _c_int, _c_vp]),
    "gguf_repack_q6k_planes": (_c_int, [_c_vp, _c_vp, _c_i64, _c_int, _c_vp]),
    "gguf_dequant_padded": (_c_int, [_c_vp, _c_int, _c_int, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp]),
    "gguf_dense_gemm": (_c_int, [_c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_vp,
                                 _c_int, _c_vp, _c_sz, _c_vp]),
    "gguf_dense_gemm_noalloc": (_c_int, [_c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp,
                                         _c_vp, _c_int, _c_vp]),
    "gguf_mm_check_errors": (_c_int, [_c_vp]),
    "gguf_mm_status_string": (ctypes.c_char_p, [_c_int]),
    "gguf_mm_version": (_c_int, []),
    "gguf_mm_debug_gemv_terms": (_c_int, [_c_vp, _c_int, _c_int, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp,
                                          _c_vp, _c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp, _c_sz, _c_int,
                                          ctypes.POINTER(_c_int), _c_vp]),
    "gguf_mm_gemv_kernel": (_c_int, [_c_int, _c_int, _c_i64, _c_i64, _c_i64, _c_int]),
    "gguf_mm_auto_path": (_c_int, [_c_int, _c_int, _c_i64, _c_i64, _c_i64, _c_int]),
    "gguf_mm_debug_moe_route": (_c_int, [_c_vp, _c_i64, _c_i64, _c_vp, _c_vp, _c_vp, _c_i64, _c_vp, _c_vp]),
    "gguf_mm_debug_timeout": (_c_int, [_c_i64, _c_vp]),
    "gguf_mm_debug_moe_mv_terms": (_c_int, [_c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp,
                                            _c_i64, _c_int, _c_vp, _c_vp, _c_int, _c_vp, _c_vp, _c_vp, _c_vp, _c_vp,
                                            _c_sz, _c_vp]),
    "gguf_file_open": (_c_int, [ctypes.c_char_p, ctypes.POINTER(_c_vp)]),
    "gguf_file_close": (None, [_c_vp]),
    "gguf_file_version": (_c_int, [_c_vp]),
    "gguf_file_alignment": (_c_i64, [_c_vp]),
    "gguf_file_tensor_count": (_c_i64, [_c_vp]),
    "gguf_file_tensor_info": (_c_int, [_c_vp, _c_i64, ctypes.c_char_p, _c_sz, ctypes.POINTER(_c_int),
                                       ctypes.POINTER(_c_int), ctypes.POINTER(_c_i64),
                                       ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]),
    "gguf_file_find_tensor": (_c_i64, [_c_vp, ctypes.c_char_p]),
    "gguf_file_read_tensor": (_c_int, [_c_vp, _c_i64, _c_vp, _c_sz]),
    "gguf_file_tensor_as_weight": (_c_int, [_c_vp, _c_i64, ctypes.POINTER(_c_int), ctypes.POINTER(_c_i64),
                                            ctypes.POINTER(_c_i64)]),
    "gguf_file_kv_count": (_c_i64, [_c_vp]),
    "gguf_file_kv_key": (_c_int, [_c_vp, _c_i64, ctypes.c_char_p, _c_sz, ctypes.POINTER(_c_int)]),
    "gguf_file_get_int": (_c_int, [_c_vp, ctypes.c_char_p, ctypes.POINTER(_c_i64)]),
    "gguf_file_get_float": (_c_int, [_c_vp, ctypes.c_char_p, ctypes.POINTER(ctypes.c_double)]),
    "gguf_file_get_string": (_c_int, [_c_vp, ctypes.c_char_p, ctypes.c_char_p, _c_sz, ctypes.POINTER(_c_sz)]),
    "gguf_file_get_array": (_c_int, [_c_vp, ctypes.c_char_p, ctypes.POINTER(_c_int), ctypes.POINTER(_c_i64),
                                     _c_vp, _c_sz]),
}

_lib = None


class GGUFError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: status {status} ({status_string(status)})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load (once) and return the shared library; raises if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise ImportError(f"{path} is missing: build it with __graft_entry__.build() "
                              "(or python gguf_quant_weight_gb300/_build.py)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def exported_symbols():
    return list(_SIGS)


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, st):
    if st != 0:
        raise GGUFError(fn, st)
    return st


def status_string(status: int) -> str:
    return load_library().gguf_mm_status_string(status).decode()


def gguf_mm_version() -> int:
    return load_library().gguf_mm_version()


def gguf_mm_workspace_size(op, qtype, N, K, M, n_expert=0, top_k=0) -> int:
    return load_library().gguf_mm_workspace_size(op, qtype, N, K, M, n_expert, top_k)


def gguf_mm_gemv(w, qtype, layout, N, K, x, xdt, M, residual, y, ydt, workspace=None, ws_bytes=0, stream=None):
    return _check("gguf_mm_gemv", load_library().gguf_mm_gemv(
        _p(w), qtype, layout, N, K, _p(x), xdt, M, _p(residual), _p(y), ydt, _p(workspace), ws_bytes, _s(stream)))


def gguf_mm_gemv_host(w, qtype, layout, N, K, x_host, x_dev, xdt, M, residual_host, residual_dev, y_host, y_dev,
                      ydt, workspace=None, ws_bytes=0, stream=None):
    return _check("gguf_mm_gemv_host", load_library().gguf_mm_gemv_host(
        _p(w), qtype, layout, N, K, _p(x_host), _p(x_dev), xdt, M, _p(residual_host), _p(residual_dev),
        _p(y_host), _p(y_dev), ydt, _p(workspace), ws_bytes, _s(stream)))


def gguf_mm_gemm(w, qtype, layout, N, K, x, xdt, M, residual, y, ydt, workspace=None, ws_bytes=0,
                 path=GGUF_PATH_AUTO, stream=None):
    return _check("gguf_mm_gemm", load_library().gguf_mm_gemm(
        _p(w), qtype, layout, N, K, _p(x), xdt, M, _p(residual), _p(y), ydt, _p(workspace), ws_bytes, path,
        _s(stream)))


def gguf_mm_id(w_experts, qtype, n_expert, N, K, x, xdt, T, ids, top_k, residual, y, ydt, workspace=None,
               ws_bytes=0, stream=None):
    return _check("gguf_mm_id", load_library().gguf_mm_id(
        _p(w_experts), qtype, n_expert, N, K, _p(x), xdt, T, _p(ids), top_k, _p(residual), _p(y), ydt,
        _p(workspace), ws_bytes, _s(stream)))


def gguf_mm_id_slots(w_experts, qtype, n_expert, N, K, x, xdt, T, ids, top_k, residual, y, ydt, workspace=None,
                     ws_bytes=0, stream=None):
    return _check("gguf_mm_id_slots", load_library().gguf_mm_id_slots(
        _p(w_experts), qtype, n_expert, N, K, _p(x), xdt, T, _p(ids), top_k, _p(residual), _p(y), ydt,
        _p(workspace), ws_bytes, _s(stream)))


def gguf_mm_id_form(qtype, T, top_k) -> int:
    return load_library().gguf_mm_id_form(qtype, T, top_k)


def gguf_mm_id_path(w_experts, qtype, n_expert, N, K, x, xdt, T, ids, top_k, per_slot, residual, y, ydt,
                    workspace=None, ws_bytes=0, path=GGUF_PATH_AUTO, stream=None):
    return _check("gguf_mm_id_path", load_library().gguf_mm_id_path(
        _p(w_experts), qtype, n_expert, N, K, _p(x), xdt, T, _p(ids), top_k, per_slot, _p(residual), _p(y), ydt,
        _p(workspace), ws_bytes, path, _s(stream)))


def gguf_repack_q6k_planes(src, dst, nblk, inverse=0, stream=None):
    return _check("gguf_repack_q6k_planes", load_library().gguf_repack_q6k_planes(
        _p(src), _p(dst), nblk, inverse, _s(stream)))


def gguf_dequant_padded(w, qtype, layout, N, K, out, odt, ld, stream=None):
    return _check("gguf_dequant_padded", load_library().gguf_dequant_padded(
        _p(w), qtype, layout, N, K, _p(out), odt, ld, _s(stream)))


def gguf_dense_gemm(wdense, wdt, ld, N, K, x, xdt, M, residual, y, ydt, workspace=None, ws_bytes=0, stream=None):
    return _check("gguf_dense_gemm", load_library().gguf_dense_gemm(
        _p(wdense), wdt, ld, N, K, _p(x), xdt, M, _p(residual), _p(y), ydt, _p(workspace), ws_bytes, _s(stream)))


def gguf_dense_gemm_noalloc(wdense, wdt, ld, N, K, x, xdt, M, residual, y, ydt, stream=None):
    return _check("gguf_dense_gemm_noalloc", load_library().gguf_dense_gemm_noalloc(
        _p(wdense), wdt, ld, N, K, _p(x), xdt, M, _p(residual), _p(y), ydt, _s(stream)))


def gguf_mm_check_errors(stream=None) -> int:
    """Returns the device status (0 or a negative code) without raising."""
    return load_library().gguf_mm_check_errors(_s(stream))


GEMV_KERNELS = {0: "staged", 1: "direct", 2: "tile", 3: "pair", 4: "rowlane"}


def gguf_mm_debug_gemv_terms(w, qtype, layout, N, K, x, xdt, M, residual, y, ydt, qa=None, d_a=None, s=None,
                             D=None, workspace=None, ws_bytes=0, kernel=-1, stream=None) -> int:
    """Runs the GEMV with its integer intermediates dumped; returns the id of the kernel that ran."""
    out = _c_int(-1)
    _check("gguf_mm_debug_gemv_terms", load_library().gguf_mm_debug_gemv_terms(
        _p(w), qtype, layout, N, K, _p(x), xdt, M, _p(residual), _p(y), ydt, _p(qa), _p(d_a), _p(s), _p(D),
        _p(workspace), ws_bytes, kernel, ctypes.byref(out), _s(stream)))
    return out.value


def gguf_mm_auto_path(qtype, layout, N, K, M, xdt=GGUF_DT_BF16) -> int:
    """The path GGUF_PATH_AUTO takes for this shape (GGUF_PATH_GEMV or GGUF_PATH_FUSED)."""
    return load_library().gguf_mm_auto_path(qtype, layout, N, K, M, xdt)


def gguf_mm_gemv_kernel(qtype, layout, N, K, M, xdt=GGUF_DT_BF16) -> int:
    """The id of the GEMV kernel gguf_mm_gemv picks for this shape (negative status on error)."""
    return load_library().gguf_mm_gemv_kernel(qtype, layout, N, K, M, xdt)


def gguf_mm_debug_moe_route(ids, entries, n_expert, offsets, ntiles, tiles, max_tiles, rows, stream=None):
    return _check("gguf_mm_debug_moe_route", load_library().gguf_mm_debug_moe_route(
        _p(ids), entries, n_expert, _p(offsets), _p(ntiles), _p(tiles), max_tiles, _p(rows), _s(stream)))


def gguf_mm_debug_moe_mv_terms(w_experts, qtype, n_expert, N, K, x, xdt, T, ids, top_k, per_slot, residual, y, ydt,
                               qa=None, d_a=None, s=None, D=None, workspace=None, ws_bytes=0, stream=None):
    return _check("gguf_mm_debug_moe_mv_terms", load_library().gguf_mm_debug_moe_mv_terms(
        _p(w_experts), qtype, n_expert, N, K, _p(x), xdt, T, _p(ids), top_k, per_slot, _p(residual), _p(y), ydt,
        _p(qa), _p(d_a), _p(s), _p(D), _p(workspace), ws_bytes, _s(stream)))


def gguf_mm_debug_timeout(spin_limit, stream=None):
    return _check("gguf_mm_debug_timeout", load_library().gguf_mm_debug_timeout(spin_limit, _s(stream)))


# --- GGUF container reader (host only) ---------------------------------------

def _enc(s):
    return s.encode("utf-8", "surrogateescape")


def _dec(b):
    return b.decode("utf-8", "surrogateescape")


class GGUFFile:
    """A .gguf file opened through gguf_file_open: metadata values and tensor bytes.

    Thin marshalling over the gguf_file_* entry points; the parsing and every
    bounds check are in the library.  `tensors()` lists (name, type, dims);
    `tensor_bytes(name)` returns the tensor's bytes as a numpy u8 array, which
    for a block-quantized weight W[N, K] is the [N, K/blk*bb] block array the
    matmul entry points take."""

    def __init__(self, path):
        self._h = None
        lib = load_library()
        h = _c_vp()
        _check("gguf_file_open", lib.gguf_file_open(os.fsencode(path), ctypes.byref(h)))
        self._h = h.value
        self._lib = lib

    def close(self):
        if getattr(self, "_h", None):
            self._lib.gguf_file_close(self._h)
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        self.close()

    @property
    def version(self) -> int:
        return self._lib.gguf_file_version(self._h)

    @property
    def alignment(self) -> int:
        return self._lib.gguf_file_alignment(self._h)

    def tensor_info(self, index):
        """(name, type, dims (contiguous first), absolute data offset, nbytes)."""
        n = 1024
        while True:
            name = ctypes.create_string_buffer(n)
            t, nd = _c_int(), _c_int()
            dims = (_c_i64 * 4)()
            off, nb = ctypes.c_uint64(), ctypes.c_uint64()
            st = self._lib.gguf_file_tensor_info(self._h, index, name, n, ctypes.byref(t), ctypes.byref(nd), dims,
                                                 ctypes.byref(off), ctypes.byref(nb))
            if st == GGUF_ERR_WORKSPACE:
                n *= 16
                continue
            _check("gguf_file_tensor_info", st)
            return _dec(name.value), t.value, tuple(dims[:nd.value]), off.value, nb.value

    def tensors(self):
        return [self.tensor_info(i)[:3] for i in range(self._lib.gguf_file_tensor_count(self._h))]

    def find_tensor(self, name) -> int:
        i = self._lib.gguf_file_find_tensor(self._h, _enc(name))
        if i < 0:
            raise GGUFError("gguf_file_find_tensor", int(i))
        return int(i)

    def tensor_bytes(self, name_or_index):
        import numpy as np
        i = self.find_tensor(name_or_index) if isinstance(name_or_index, str) else name_or_index
        nb = self.tensor_info(i)[4]
        out = np.empty(nb, np.uint8)
        _check("gguf_file_read_tensor", self._lib.gguf_file_read_tensor(self._h, i, out.ctypes.data, nb))
        return out

    def weight(self, name):
        """(blocks as a [N, row_bytes] u8 array, qtype, N, K) of a 2-D block-quantized tensor."""
        i = self.find_tensor(name)
        qt, n, k = _c_int(), _c_i64(), _c_i64()
        _check("gguf_file_tensor_as_weight", self._lib.gguf_file_tensor_as_weight(
            self._h, i, ctypes.byref(qt), ctypes.byref(n), ctypes.byref(k)))
        return self.tensor_bytes(i).reshape(n.value, -1), qt.value, n.value, k.value

    def keys(self):
        out = []
        for i in range(self._lib.gguf_file_kv_count(self._h)):
            n = 256
            while True:
                buf, vt = ctypes.create_string_buffer(n), _c_int()
                st = self._lib.gguf_file_kv_key(self._h, i, buf, n, ctypes.byref(vt))
                if st == GGUF_ERR_WORKSPACE:
                    n *= 16
                    continue
                _check("gguf_file_kv_key", st)
                out.append((_dec(buf.value), vt.value))
                break
        return out

    def get_int(self, key) -> int:
        v = _c_i64()
        _check("gguf_file_get_int", self._lib.gguf_file_get_int(self._h, _enc(key), ctypes.byref(v)))
        return v.value

    def get_float(self, key) -> float:
        v = ctypes.c_double()
        _check("gguf_file_get_float", self._lib.gguf_file_get_float(self._h, _enc(key), ctypes.byref(v)))
        return v.value

    def get_string(self, key) -> str:
        n = _c_sz()
        _check("gguf_file_get_string", self._lib.gguf_file_get_string(self._h, _enc(key), None, 0,
                                                                      ctypes.byref(n)))
        buf = ctypes.create_string_buffer(n.value + 1)
        _check("gguf_file_get_string", self._lib.gguf_file_get_string(self._h, _enc(key), buf, n.value + 1,
                                                                      None))
        return _dec(buf.raw[:n.value])

    _ARRAY_NP = {0: "u1", 1: "i1", 2: "<u2", 3: "<i2", 4: "<u4", 5: "<i4", 6: "<f4", 7: "u1", 10: "<u8",
                 11: "<i8", 12: "<f8"}

    def get_array(self, key):
        """A scalar array as numpy; a string array as (8, count)."""
        import numpy as np
        et, cnt = _c_int(), _c_i64()
        _check("gguf_file_get_array", self._lib.gguf_file_get_array(self._h, _enc(key), ctypes.byref(et),
                                                                    ctypes.byref(cnt), None, 0))
        if et.value not in self._ARRAY_NP:
            return et.value, cnt.value
        out = np.empty(cnt.value, self._ARRAY_NP[et.value])
        _check("gguf_file_get_array", self._lib.gguf_file_get_array(self._h, _enc(key), None, None,
                                                                    out.ctypes.data, out.nbytes))
        return out


def raw_status(fn_name: str, *args) -> int:
    """Call a C entry point with raw arguments and return its status (tests of argument checks)."""
    return getattr(load_library(), fn_name)(*args)
