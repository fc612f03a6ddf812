"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module only draws random numbers and lays them into the GGUF byte-block
structs; it holds none of the dequantization or matmul arithmetic, so both the
CPU oracle and the CUDA path can be fed from it without sharing any method code.

Block structs (byte offsets inside one block) follow the GGUF on-disk layout:

  Q4_0  18 B / 32 values : d f16 @0, qs[16] @2 (element e < 16: low nibble of qs[e], else high of qs[e-16])
  Q4_1  20 B / 32 values : d f16 @0, m f16 @2, qs[16] @4
  Q5_0  22 B / 32 values : d f16 @0, qh[4] @2 (bit e: fifth bit of element e), qs[16] @6
  Q5_1  24 B / 32 values : d f16 @0, m f16 @2, qh[4] @4, qs[16] @8

  Q2_K  84 B / 256 values: scales[16] @0 (scale | min << 4), qs[64] @16, d f16 @80, dmin f16 @82
  Q3_K 110 B / 256 values: hmask[32] @0, qs[64] @32, scales[12] @96, d f16 @108

  Q8_0  34 B / 32 values : d f16 @0, qs[32] i8 @2
  Q4_K 144 B / 256 values: d f16 @0, dmin f16 @2, scales[12] @4, qs[128] @16
  Q5_K 176 B / 256 values: d f16 @0, dmin f16 @2, scales[12] @4, qh[32] @16, qs[128] @48
  Q6_K 210 B / 256 values: ql[128] @0, qh[64] @128, scales[16] i8 @192, d f16 @208

(GGUF Support Proposal for mobius, section 7 "Quantization Format Deep Dive" and the
section 1.2 type table; Q5_K/Q6_K field sizes from OpenVINO PR #39119,
"Transformation", where the Q6_K plane list names ql/qh/scales/d sizes.)

Recipes (one per workload family, all N(0,1)/uniform draws from numpy PCG64):
  * Q6_K: ql/qh uniform bytes, scales uniform integers in [-32, 31], d = f16(|N(0,1)|*1e-3)
  * Q5_K / Q4_K: qs/qh/scales uniform bytes, d and dmin = f16(|N(0,1)|*1e-3)
  * Q8_0: q uniform integers in [-127, 127], d = f16(|N(0,1)|*1e-3)
  * Q4_0 / Q5_0: qs/qh uniform bytes, d = f16(|N(0,1)|*1e-3)
  * Q4_1 / Q5_1: as Q4_0 / Q5_0, plus m = f16(-8e-3 * |N(0,1)| * (1 + |N(0,1)|))
  * Q2_K: scales/qs uniform bytes, d and dmin = f16(|N(0,1)|*1e-3)
  * Q3_K: hmask/qs/scales uniform bytes, d = f16(|N(0,1)|*1e-3)
  * activations and residuals: N(0,1), kept as f32 or rounded to bf16/f16
  * MoE ids: per token top_k distinct experts drawn in turn without replacement,
    P(rank r) proportional to r**-s over ranks 1..n_expert, expert id = rank - 1
"""
from __future__ import annotations

import numpy as np

Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K = 2, 3, 6, 7, 8, 12, 13, 14
Q2_K, Q3_K = 10, 11
QTYPE_NAMES = {Q4_0: "Q4_0", Q4_1: "Q4_1", Q5_0: "Q5_0", Q5_1: "Q5_1", Q8_0: "Q8_0", Q2_K: "Q2_K", Q3_K: "Q3_K",
               Q4_K: "Q4_K", Q5_K: "Q5_K", Q6_K: "Q6_K"}
BLOCK_VALUES = {Q4_0: 32, Q4_1: 32, Q5_0: 32, Q5_1: 32, Q8_0: 32, Q2_K: 256, Q3_K: 256, Q4_K: 256, Q5_K: 256,
                Q6_K: 256}
BLOCK_BYTES = {Q4_0: 18, Q4_1: 20, Q5_0: 22, Q5_1: 24, Q8_0: 34, Q2_K: 84, Q3_K: 110, Q4_K: 144, Q5_K: 176,
               Q6_K: 210}


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def row_bytes(qtype: int, K: int) -> int:
    return K // BLOCK_VALUES[qtype] * BLOCK_BYTES[qtype]


def _f16_scale_bytes(g: np.random.Generator, n: int) -> np.ndarray:
    """n little-endian f16 values |N(0,1)|*1e-3, as a [n, 2] u8 array."""
    v = (np.abs(g.standard_normal(n)) * 1e-3).astype(np.float16)
    return v.view(np.uint8).reshape(n, 2)


def weight_blocks(g: np.random.Generator, qtype: int, N: int, K: int) -> np.ndarray:
    """Random weight tensor in GGUF byte blocks, shape [N, row_bytes] u8."""
    bv, bb = BLOCK_VALUES[qtype], BLOCK_BYTES[qtype]
    if K % bv:
        raise ValueError(f"K={K} is not a multiple of {bv}")
    nb = N * (K // bv)
    blk = g.integers(0, 256, size=(nb, bb), dtype=np.uint8)
    if qtype == Q8_0:
        blk[:, 0:2] = _f16_scale_bytes(g, nb)
        blk[:, 2:34] = g.integers(-127, 128, size=(nb, 32), dtype=np.int8).view(np.uint8)
    elif qtype in (Q4_K, Q5_K):
        blk[:, 0:2] = _f16_scale_bytes(g, nb)
        blk[:, 2:4] = _f16_scale_bytes(g, nb)
    elif qtype == Q6_K:
        blk[:, 192:208] = g.integers(-32, 32, size=(nb, 16), dtype=np.int8).view(np.uint8)
        blk[:, 208:210] = _f16_scale_bytes(g, nb)
    elif qtype in (Q4_0, Q5_0):
        blk[:, 0:2] = _f16_scale_bytes(g, nb)
    elif qtype == Q2_K:
        blk[:, 80:82] = _f16_scale_bytes(g, nb)
        blk[:, 82:84] = _f16_scale_bytes(g, nb)
    elif qtype == Q3_K:
        blk[:, 108:110] = _f16_scale_bytes(g, nb)
    elif qtype in (Q4_1, Q5_1):
        blk[:, 0:2] = _f16_scale_bytes(g, nb)
        # the min: m = -8 * |N(0,1)| * 1e-3 * (1 + |N(0,1)|), negative like a block's smallest weight
        mv = (-8e-3 * np.abs(g.standard_normal(nb)) * (1 + np.abs(g.standard_normal(nb)))).astype(np.float16)
        blk[:, 2:4] = mv.view(np.uint8).reshape(nb, 2)
    else:
        raise ValueError(f"unknown qtype {qtype}")
    return np.ascontiguousarray(blk.reshape(N, -1))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round f32 to bf16 (nearest, ties to even) and return the u16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def normal(g: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0,1) samples: dtype 'f32' -> float32; 'bf16' -> u16 bits; 'f16' -> float16."""
    a = g.standard_normal(shape).astype(np.float32)
    if dtype == "f32":
        return a
    if dtype == "bf16":
        return f32_to_bf16_bits(a)
    if dtype == "f16":
        return a.astype(np.float16)
    raise ValueError(dtype)


def zipf_ids(g: np.random.Generator, T: int, n_expert: int, top_k: int, s: float = 1.1) -> np.ndarray:
    """[T, top_k] int32 expert ids, distinct within a token, Zipf(s) over rank."""
    p = np.arange(1, n_expert + 1, dtype=np.float64) ** (-s)
    ids = np.empty((T, top_k), dtype=np.int32)
    for t in range(T):
        w = p.copy()
        for k in range(top_k):
            e = g.choice(n_expert, p=w / w.sum())
            ids[t, k] = e
            w[e] = 0.0
    return ids


# Workload shapes (one entry per benchmark family).
CONFIGS = {
    "q6k_gemv_256x1024": dict(seed=1000, qtype=Q6_K, N=256, K=1024, M=[1], xdt="f32", ydt="f32"),
    "q5k_gemv_4096x4096_res": dict(seed=1001, qtype=Q5_K, N=4096, K=4096, M=[1, 2, 4], xdt="bf16",
                                   ydt="bf16", residual=True),
    "q6k_q5k_gemm_14336x4096": dict(seed=1002, qtypes=[Q6_K, Q5_K], N=14336, K=4096,
                                    M=[8, 64, 128, 256, 512, 2048], xdt="bf16", ydt="bf16"),
    "q8_0_gemm_2048x8192": dict(seed=1003, qtype=Q8_0, N=2048, K=8192, M=[128, 512, 4096],
                                xdt="bf16", ydt="bf16"),
    "q4k_moe_128x768x2048_top8": dict(seed=1004, qtype=Q4_K, n_expert=128, top_k=8, N=768, K=2048,
                                      T=[32, 64, 256, 512], xdt="bf16", ydt="bf16", zipf_s=1.1),
}
