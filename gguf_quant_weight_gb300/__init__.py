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
GGUF_Q8_0, GGUF_Q4_K, GGUF_Q5_K, GGUF_Q6_K = 8, 12, 13, 14
GGUF_LAYOUT_BLOCKS, GGUF_LAYOUT_Q6K_PLANES = 0, 1
GGUF_DT_F32, GGUF_DT_F16, GGUF_DT_BF16 = 0, 1, 2
GGUF_PATH_AUTO, GGUF_PATH_GEMV, GGUF_PATH_FUSED = 0, 1, 2
GGUF_OP_GEMV, GGUF_OP_GEMM, GGUF_OP_ID, GGUF_OP_DENSE = 0, 1, 2, 3
GGUF_OK = 0
GGUF_ERR_INVALID_ARG, GGUF_ERR_UNSUPPORTED, GGUF_ERR_MISALIGNED = -1, -2, -3
GGUF_ERR_WORKSPACE, GGUF_ERR_CUDA, GGUF_ERR_TIMEOUT, GGUF_ERR_NO_DEVICE = -4, -5, -6, -7

BLOCK_VALUES = {GGUF_Q8_0: 32, GGUF_Q4_K: 256, GGUF_Q5_K: 256, GGUF_Q6_K: 256}
BLOCK_BYTES = {GGUF_Q8_0: 34, GGUF_Q4_K: 144, GGUF_Q5_K: 176, GGUF_Q6_K: 210}

_c_i64, _c_int, _c_sz, _c_vp = ctypes.c_int64, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p

# name -> (restype, argtypes); mirrors include/gguf_mm.h
_SIGS = {
    "gguf_mm_workspace_size": (_c_sz, [_c_int, _c_int, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64]),
    "gguf_mm_gemv": (_c_int, [_c_vp, _c_int, _c_int, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_vp,
                              _c_int, _c_vp, _c_sz, _c_vp]),
    "gguf_mm_gemm": (_c_int, [_c_vp, _c_int, _c_int, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_vp,
                              _c_int, _c_vp, _c_sz, _c_int, _c_vp]),
    "gguf_mm_id": (_c_int, [_c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_i64,
                            _c_vp, _c_vp, _c_int, _c_vp, _c_sz, _c_vp]),
    "gguf_mm_id_slots": (_c_int, [_c_vp, _c_int, _c_i64, _c_i64, _c_i64, _c_vp, _c_int, _c_i64, _c_vp, _c_i64,
                                  _c_vp, _c_vp, _c_int, _c_vp, _c_sz, _c_vp]),
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


def gguf_mm_debug_timeout(spin_limit, stream=None):
    return _check("gguf_mm_debug_timeout", load_library().gguf_mm_debug_timeout(spin_limit, _s(stream)))


def raw_status(fn_name: str, *args) -> int:
    """Call a C entry point with raw arguments and return its status (tests of argument checks)."""
    return getattr(load_library(), fn_name)(*args)
