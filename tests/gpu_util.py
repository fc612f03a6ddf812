"""Helpers for the GPU parity tests: device copies of numpy inputs and the
tolerance rules used throughout.

Tolerances (floating-point outputs):
  * f32 output:        max |got - ref| <= 1e-4 * max |ref|
  * bf16 / f16 output: max (|got - ref| - ulp_out(ref)/2) <= 2e-3 * max |ref|
    (rounding the result to the output type alone can move it by half an ulp,
    so that half ulp is granted per element on top of the bound)
Integer, byte and index results are compared exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import gguf_quant_weight_gb300 as g

DT = {"f32": g.GGUF_DT_F32, "f16": g.GGUF_DT_F16, "bf16": g.GGUF_DT_BF16}
TORCH_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


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


def half_ulp(ref: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.zeros_like(ref)
    mant = 7 if dtype == "bf16" else 10
    e = np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -24)))
    return 0.5 * 2.0 ** (e - mant)


def check_close(got: np.ndarray, ref: np.ndarray, out_dtype: str, rel: float | None = None, what: str = ""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    scale = np.max(np.abs(ref))
    if rel is None:
        rel = 1e-4 if out_dtype == "f32" else 2e-3
    excess = np.abs(got - ref) - half_ulp(ref, out_dtype)
    worst = float(np.max(excess)) if excess.size else 0.0
    assert worst <= rel * scale, f"{what}: max excess err {worst:.3e} > {rel:.1e} * {scale:.3e}"
    return worst / scale if scale else 0.0


def require_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    g.load_library()


def gemv_workspace(M: int, K: int):
    """A device workspace for gguf_mm_gemv of M rows of K values: (tensor, bytes)."""
    import gguf_quant_weight_gb300 as g
    n = g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, 0, 1, K, M)
    return torch.empty(max(n, 256), dtype=torch.uint8, device="cuda"), n
