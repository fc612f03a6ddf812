"""Helpers for the GPU parity tests: device copies of numpy inputs, guarded
output buffers and the tolerance rules used throughout.

Tolerances (floating-point outputs; integer, byte and index results are
compared exactly):
  * f32 output: max |got - ref| <= rel * max |ref|, rel = 1e-4 for the int8
    GEMV path and 2e-3 for the f16 tensor-core paths.  Nothing is granted for
    rounding: f32's own rounding (2**-24) is far below both bounds.
  * bf16 / f16 output: every element must be the output type's rounding of a
    value within 2e-3 * max |ref| of the oracle -- the distance from ref to the
    interval of reals that round to `got` is at most 2e-3 * max |ref|.  This is
    the bound on the arithmetic with only the final rounding of the stored
    value set aside.  (A check of |got - round(ref)| would fail whenever the
    exact result and ref fall on two sides of a rounding boundary: one bf16
    ulp in the top binade is 4e-3 to 8e-3 of max |ref|, twice the bound.)
    Every path is also tested with f32 output, where the bound holds raw.

Guard zones: outputs and workspaces are allocated with 4 KiB of canary bytes on
both sides (the stand-in for a memory sanitizer on this pool); every helper
that launches checks that the canaries are intact afterwards.
"""
from __future__ import annotations

import numpy as np
import torch

import gguf_quant_weight_gb300 as g

DT = {"f32": g.GGUF_DT_F32, "f16": g.GGUF_DT_F16, "bf16": g.GGUF_DT_BF16}
TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
GUARD = 4096
CANARY = 0xA5


def dev(a: np.ndarray, dtype: str | None = None) -> torch.Tensor:
    """numpy -> cuda tensor; bf16 arrays are passed as u16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(a)).to("cuda")
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    return t


def host64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def act_f32(a: np.ndarray, dtype: str) -> np.ndarray:
    """The f32 value of an activation array as the kernels read it."""
    from oracle import gguf_oracle as O
    if dtype == "bf16":
        return O.bf16_bits_to_f32(a)
    return np.asarray(a, dtype=np.float32)


def act_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    return act_f32(a, dtype).astype(np.float64)


# ---------------------------------------------------------------- guard zones

class Guarded:
    """A device buffer of `shape` x `dtype` with GUARD canary bytes before and after it."""

    def __init__(self, shape, dtype: torch.dtype, fill=None):
        shape = tuple(int(s) for s in (shape if isinstance(shape, (tuple, list)) else (shape,)))
        esize = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape)) if shape else 1
        self.nbytes = n * esize
        self.raw = torch.full((GUARD + self.nbytes + GUARD,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self, what: str = ""):
        torch.cuda.synchronize()
        head = self.raw[:GUARD].cpu().numpy()
        tail = self.raw[GUARD + self.nbytes:].cpu().numpy()
        bad_h = np.flatnonzero(head != CANARY)
        bad_t = np.flatnonzero(tail != CANARY)
        assert bad_h.size == 0, f"{what}: write {GUARD - bad_h[0]} bytes before the buffer"
        assert bad_t.size == 0, f"{what}: write {bad_t[0]} bytes past the end of the buffer"


def guarded(shape, dtype: torch.dtype, fill=None) -> Guarded:
    return Guarded(shape, dtype, fill)


def workspace(nbytes: int, fill: int = 0) -> Guarded:
    """A guarded device workspace of nbytes (at least 16) bytes, every byte = fill."""
    return Guarded((max(int(nbytes), 16),), torch.uint8, fill)


# ---------------------------------------------------------------- tolerances

def _rounding_interval(got: np.ndarray, dtype: str):
    """Lower and upper ends of the interval of reals that round (to nearest) to
    each element of `got`, which holds values of the bf16 / f16 type."""
    mant, emin = (7, -126) if dtype == "bf16" else (10, -14)
    a = np.abs(got)
    e = np.where(a > 0, np.floor(np.log2(np.where(a > 0, a, 1.0))), emin)
    e = np.maximum(e, emin)                                   # subnormals share the smallest spacing
    ulp = np.ldexp(1.0, (e - mant).astype(np.int64))
    below = np.where((a == np.ldexp(1.0, e.astype(np.int64))) & (e > emin), ulp / 2, ulp)  # binade bottom
    below = np.where(a == 0, ulp, below)
    toward0, away = below / 2, ulp / 2                        # half-gaps to the neighbours
    lo = np.where(got >= 0, got - toward0, got - away)
    hi = np.where(got >= 0, got + away, got + toward0)
    lo = np.where(got == 0, -ulp / 2, lo)
    return lo, hi


def check_close(got: np.ndarray, ref: np.ndarray, out_dtype: str, rel: float | None = None, what: str = "",
                allow_nan: bool = False):
    """Asserts the tolerance rule of the module docstring; returns the worst
    error as a fraction of max |ref|.  allow_nan: NaN must appear exactly
    where ref is NaN (and is then not compared)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if allow_nan:
        assert np.array_equal(np.isnan(got), np.isnan(ref)), f"{what}: NaN positions differ"
        keep = ~np.isnan(ref)
        got, ref = got[keep], ref[keep]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if got.size == 0:
        return 0.0
    scale = np.max(np.abs(ref))
    if rel is None:
        rel = 1e-4 if out_dtype == "f32" else 2e-3
    if out_dtype == "f32":
        err = np.abs(got - ref)
    else:
        lo, hi = _rounding_interval(got, out_dtype)
        err = np.maximum(np.maximum(lo - ref, ref - hi), 0.0)
    worst = float(np.max(err))
    assert worst <= rel * scale, f"{what}: max err {worst:.3e} > {rel:.1e} * {scale:.3e}"
    return worst / scale if scale else 0.0


def require_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.load_library()


def gemv_workspace(M: int, K: int):
    """A device workspace for gguf_mm_gemv of M rows of K values: (tensor, bytes)."""
    n = g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, 0, 1, K, M)
    return torch.empty(max(n, 256), dtype=torch.uint8, device="cuda"), n


def moe_mv_max_rows(qtype: int) -> int:
    """Routed rows (T * top_k) up to which gguf_mm_id takes its decode form (one
    int8 GEMV per routed row), as the library's header states it."""
    if qtype in (g.GGUF_Q4_K, g.GGUF_Q5_K, g.GGUF_Q2_K, g.GGUF_Q3_K, g.GGUF_Q6_K):
        return 128
    return 16 if qtype == g.GGUF_Q8_0 else 32


def moe_decode_form(qtype: int, entries: int) -> bool:
    return entries <= moe_mv_max_rows(qtype)
