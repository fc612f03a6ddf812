"""CPU oracle for matmul on GGUF block-quantized weights.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
cpu_baseline / reference legs of bench.py may import or run this module.  The
product path (the CUDA library and its Python binding) never calls it, and this
module imports nothing from the product package.

Plain numpy, float64 for every floating-point result, written for a reader to
check against the sources by eye: no blocking, fusion or reordering beyond what
each definition states.  A library primitive (numpy matmul) is the only
shortcut.

Sources (web pages; cited by title and section):
  [mobius]  "GGUF Support Proposal for mobius": section 1.2 "Quantization Types"
            (type table: Q4_0 .. Q8_0, Q2_K .. Q6_K), section 7 "Quantization
            Format Deep Dive" (7.1 Q4_0, 7.2 Q4_1, 7.3 Q4_K, 7.4 Q8_0 block
            structs and their dequantization formulas).
  [ov39119] OpenVINO PR #39119 "FullyConnectedGGUF": "Transformation" (Q6_K plane
            regrouping QL|QH|SC|D), "Implementation" (GEMV: activations quantized
            per 32 values, int8 dot products against the blocks).
  [ov38696] OpenVINO PR #38696 (exact zero points), "Details": w = d*q - m for
            Q4_K/Q5_K, the min applied exactly (never rounded into an integer zp).
  [rocm37]  ROCm llama.cpp PR #37 "one-time K-padded f16 dequantization for
            prefill GEMMs": "How it works" (row stride padded by one cache line),
            "Correctness" (padding changes only the stride).
  [ll28301] llama.cpp PR #28301 "metal : skip the empty half of the mul_mm_id
            token tile": "Overview" (mul_mm_id: each routed (token, slot) row
            multiplies one expert's weight).

Readings taken where the pages are silent (all listed in the design notes):
  * bit packing of ql/qh/qs/scales inside each block: the GGUF on-disk layout
    (the pages' purpose is running real GGUF files); 6-bit sub-scale/min field
    order as in decode_6bit below;
  * activation quantizer rounding: f32 d_a = amax/127, multiply by f32 1/d_a,
    clamp to [-127, 127], round half away from zero; zero block -> d_a = 0;
  * a Q6_K 16-wide sub-block uses the activation block floor(j/2), and so do the
    16-value sub-blocks of Q2_K and Q3_K;
  * the 32-value formats: element e < 16 in the low nibble of qs[e], e >= 16 in
    the high nibble of qs[e-16], Q5_0/Q5_1's fifth bit bit e of the qh word;
    zero points 8 (Q4_0) and 16 (Q5_0); Q4_1/Q5_1 add the min (w = q*d + m, as
    mobius 7.2 writes it) where the K-quants subtract it;
  * Q2_K / Q3_K (named in the type table only): the GGUF on-disk structs, with
    Q3_K's q3 = q2 - 4 where the element's hmask bit is clear;
  * K-padding: one 128-byte line, i.e. 64 two-byte elements, pad written as 0.
Parity against real GGUF files is unpinned: no GGUF file or reference
implementation is available to this build.
"""
from __future__ import annotations

import numpy as np

Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K = 2, 3, 6, 7, 8, 12, 13, 14   # GGUF type ids
Q2_K, Q3_K = 10, 11
BLOCK_VALUES = {Q4_0: 32, Q4_1: 32, Q5_0: 32, Q5_1: 32, Q8_0: 32, Q2_K: 256, Q3_K: 256, Q4_K: 256, Q5_K: 256,
                Q6_K: 256}
BLOCK_BYTES = {Q4_0: 18, Q4_1: 20, Q5_0: 22, Q5_1: 24, Q8_0: 34, Q2_K: 84, Q3_K: 110, Q4_K: 144, Q5_K: 176,
               Q6_K: 210}


# ----------------------------------------------------------------------------
# scalar conversions
# ----------------------------------------------------------------------------

def f16_field(b: np.ndarray) -> np.ndarray:
    """Little-endian f16 stored in two bytes (last axis) -> float64, exactly."""
    b = np.ascontiguousarray(b, dtype=np.uint8)
    return b.view(np.float16)[..., 0].astype(np.float64)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (u16) -> float64, exactly (bf16 is the top half of f32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32)


def round_f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 to the nearest bf16 (ties to even), directly from the f64 value.

    bf16 has 8 significant bits.  For finite normal values the result is the
    multiple of 2**(e-7) nearest v, where 2**e <= |v| < 2**(e+1); np.rint rounds
    ties to even.  Values beyond the bf16 range are not expected here.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.array(v * 0.0)                       # zeros that keep v's sign (IEEE: rounding -0 gives -0)
    nz = v != 0
    _, ex = np.frexp(v[nz])                       # |v| = m * 2**ex, 0.5 <= m < 1
    e = np.maximum(ex - 1, -126)                  # bf16 subnormal spacing 2**-133
    q = np.ldexp(1.0, e - 7)
    r = np.rint(v[nz] / q) * q                    # v/q is exact: power-of-two divide
    out[nz] = r
    f32 = out.astype(np.float32)                  # exact: r has <= 9 significant bits
    bits = (f32.view(np.uint32) >> 16).astype(np.uint16)
    return bits


def round_f64_to_f16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 to the nearest f16, ties to even (numpy converts f64->f16 directly)."""
    return np.asarray(v, dtype=np.float64).astype(np.float16).view(np.uint16)


# ----------------------------------------------------------------------------
# per-format block decoders  ->  float64 weights
# ----------------------------------------------------------------------------

def decode_6bit(s: np.ndarray, i: int) -> np.ndarray:
    """Field i (0..15) of the 12-byte K-quant scales array: fields 0..7 are the
    sub-block scales sc_0..sc_7, fields 8..15 the sub-block mins m_0..m_7
    ([mobius] 7.3 writes sub_scale = decode_6bit(scales, j), sub_min =
    decode_6bit(scales, j + 8)).  Bit placement (reading: GGUF on-disk packing):
      j < 4 : sc_j = low 6 bits of byte j,      m_j = low 6 bits of byte j+4
      j >= 4: sc_j = low nibble of byte j+4 | top 2 bits of byte j-4 << 4
              m_j  = high nibble of byte j+4 | top 2 bits of byte j   << 4
    s: [..., 12] u8; returns an int64 array over the leading axes.
    """
    s = s.astype(np.int64)
    j, is_min = i % 8, i >= 8
    if j < 4:
        return s[..., j + 4 * is_min] & 63
    low = (s[..., j + 4] >> 4) if is_min else (s[..., j + 4] & 15)
    high = s[..., j - 4 + 4 * is_min] >> 6
    return low | (high << 4)


def dequant_q8_0(blk: np.ndarray) -> np.ndarray:
    """[nb, 34] u8 -> [nb, 32] f64.  w = d * q, q the signed byte ([mobius] 7.4, 1.2)."""
    d = f16_field(blk[:, 0:2])
    q = blk[:, 2:34].view(np.int8).astype(np.float64)
    return d[:, None] * q


def q4k_nibble(qs: np.ndarray, e: int) -> np.ndarray:
    """4-bit value of element e (0..255) of a Q4_K/Q5_K super-block: elements
    come in 4 groups of 64; group p uses bytes qs[32p .. 32p+31], the low nibble
    for its first 32 elements and the high nibble for the next 32."""
    p, r = divmod(e, 64)
    byte = qs[:, 32 * p + r % 32].astype(np.int64)
    return (byte & 15) if r < 32 else (byte >> 4)


def dequant_q4_k(blk: np.ndarray) -> np.ndarray:
    """[nb, 144] u8 -> [nb, 256] f64.  w = d*sc_j*q - dmin*m_j, j = e // 32
    ([mobius] 7.3 struct and dequantization; [ov38696] min subtracted exactly)."""
    d, dmin = f16_field(blk[:, 0:2]), f16_field(blk[:, 2:4])
    s, qs = blk[:, 4:16], blk[:, 16:144]
    out = np.empty((blk.shape[0], 256), dtype=np.float64)
    for e in range(256):
        j = e // 32
        sc, m = decode_6bit(s, j), decode_6bit(s, j + 8)
        out[:, e] = d * sc * q4k_nibble(qs, e) - dmin * m
    return out


def dequant_q5_k(blk: np.ndarray) -> np.ndarray:
    """[nb, 176] u8 -> [nb, 256] f64.  q5 = nibble + 16 * bit (e // 32) of qh[e % 32];
    w = d*sc_j*q5 - dmin*m_j ([mobius] 1.2: 5-bit K-quant; [ov38696] w = d*q - m)."""
    d, dmin = f16_field(blk[:, 0:2]), f16_field(blk[:, 2:4])
    s, qh, qs = blk[:, 4:16], blk[:, 16:48], blk[:, 48:176]
    out = np.empty((blk.shape[0], 256), dtype=np.float64)
    for e in range(256):
        j = e // 32
        hi = (qh[:, e % 32].astype(np.int64) >> j) & 1
        q5 = q4k_nibble(qs, e) + 16 * hi
        out[:, e] = d * decode_6bit(s, j) * q5 - dmin * decode_6bit(s, j + 8)
    return out


def q6k_q6(ql: np.ndarray, qh: np.ndarray, e: int) -> np.ndarray:
    """Unsigned 6-bit value of element e of a Q6_K super-block.  Two halves of
    128; in half h, element r = 32g + l (g = 0..3) takes its low 4 bits from
    ql[64h + 32(g & 1) + l] (low nibble for g < 2, high for g >= 2) and its top
    2 bits from bits 2g..2g+1 of qh[32h + l]."""
    h, r = divmod(e, 128)
    g, l = divmod(r, 32)
    b = ql[:, 64 * h + 32 * (g & 1) + l].astype(np.int64)
    lo = (b & 15) if g < 2 else (b >> 4)
    hi = (qh[:, 32 * h + l].astype(np.int64) >> (2 * g)) & 3
    return lo | (hi << 4)


def dequant_q6_k_fields(ql, qh, sc, d) -> np.ndarray:
    """Q6_K from its four fields: ql [nb,128] u8, qh [nb,64] u8, sc [nb,16] u8
    (read as i8), d [nb] f64.  w = d * scales[e // 16] * (q6 - 32)."""
    sc = sc.view(np.int8).astype(np.float64)
    out = np.empty((ql.shape[0], 256), dtype=np.float64)
    for e in range(256):
        out[:, e] = d * sc[:, e // 16] * (q6k_q6(ql, qh, e) - 32)
    return out


def dequant_q6_k(blk: np.ndarray) -> np.ndarray:
    """[nb, 210] u8 -> [nb, 256] f64 (field sizes from [ov39119] Transformation)."""
    return dequant_q6_k_fields(blk[:, 0:128], blk[:, 128:192], blk[:, 192:208],
                               f16_field(blk[:, 208:210]))


# ---- the 32-value formats of the type table ([mobius] 1.2; 7.1 Q4_0, 7.2 Q4_1)

def b32_nibble(qs: np.ndarray, e: int) -> np.ndarray:
    """4-bit code of element e (0..31) of a 32-value block whose 16 code bytes are
    qs [nb, 16]: elements 0..15 are the low nibbles of qs[0..15], elements 16..31
    the high nibbles (reading: GGUF on-disk order)."""
    byte = qs[:, e % 16].astype(np.int64)
    return (byte & 15) if e < 16 else (byte >> 4)


def b32_fifth_bit(qh: np.ndarray, e: int) -> np.ndarray:
    """Fifth bit of element e of a Q5_0 / Q5_1 block: bit e of the 32-bit
    little-endian word qh [nb, 4] (reading: GGUF on-disk layout)."""
    return (qh[:, e // 8].astype(np.int64) >> (e % 8)) & 1


def dequant_q4_0(blk: np.ndarray) -> np.ndarray:
    """[nb, 18] u8 {d f16, qs[16]} -> [nb, 32] f64.  w = (q - 8) * d ([mobius] 7.1:
    unsigned codes 0..15 recentred by the implicit zero point 8)."""
    d, qs = f16_field(blk[:, 0:2]), blk[:, 2:18]
    return np.stack([(b32_nibble(qs, e) - 8) * d for e in range(32)], axis=1)


def dequant_q4_1(blk: np.ndarray) -> np.ndarray:
    """[nb, 20] u8 {d f16, m f16, qs[16]} -> [nb, 32] f64.  w = q * d + m
    ([mobius] 7.2 writes the min added: x = qs * d + m)."""
    d, m, qs = f16_field(blk[:, 0:2]), f16_field(blk[:, 2:4]), blk[:, 4:20]
    return np.stack([b32_nibble(qs, e) * d + m for e in range(32)], axis=1)


def dequant_q5_0(blk: np.ndarray) -> np.ndarray:
    """[nb, 22] u8 {d f16, qh[4], qs[16]} -> [nb, 32] f64.  q5 = nibble + 16 * bit e
    of qh; w = (q5 - 16) * d ([mobius] 1.2: symmetric 5-bit, block 32; the
    implicit zero point is 16, half the code range, as 8 is for Q4_0)."""
    d, qh, qs = f16_field(blk[:, 0:2]), blk[:, 2:6], blk[:, 6:22]
    return np.stack([(b32_nibble(qs, e) + 16 * b32_fifth_bit(qh, e) - 16) * d for e in range(32)], axis=1)


def dequant_q5_1(blk: np.ndarray) -> np.ndarray:
    """[nb, 24] u8 {d f16, m f16, qh[4], qs[16]} -> [nb, 32] f64.  w = q5 * d + m
    ([mobius] 1.2: asymmetric 5-bit + min, the Q4_1 rule with a fifth bit)."""
    d, m, qh, qs = f16_field(blk[:, 0:2]), f16_field(blk[:, 2:4]), blk[:, 4:8], blk[:, 8:24]
    return np.stack([(b32_nibble(qs, e) + 16 * b32_fifth_bit(qh, e)) * d + m for e in range(32)], axis=1)


# ---- the 2- and 3-bit K-quants of the type table ([mobius] 1.2: Q2_K "K-quant
# super-blocks, mixed", Q3_K "3-bit dominant"; 256 values, 16 sub-blocks of 16).
# The pages give neither struct; the readings (GGUF on-disk layout) are:
#   Q2_K 84 B  {scales[16] @0, qs[64] @16, d f16 @80, dmin f16 @82}
#              scales byte j: low nibble = sub-block scale, high nibble = min;
#              w = d * (scales[j] & 15) * q2 - dmin * (scales[j] >> 4)
#   Q3_K 110 B {hmask[32] @0, qs[64] @32, scales[12] @96, d f16 @108}
#              q3 = q2 - 4 when the element's hmask bit is clear, else q2;
#              w = d * (scale6_j - 32) * q3
# with the 2-bit codes laid out alike in both (k2_position).

def k2_position(e: int):
    """(byte of qs, bit shift) of the 2-bit code of element e (0..255) of a
    Q2_K / Q3_K super-block: two halves of 128; in half h, element
    r = 32j + 16p + l (j = 0..3, p = 0..1, l = 0..15) is bits 2j..2j+1 of
    qs[32h + 16p + l].  Its sub-block (scale) is e // 16."""
    h, r = divmod(e, 128)
    j, r2 = divmod(r, 32)
    p, l = divmod(r2, 16)
    return 32 * h + 16 * p + l, 2 * j


def q2_code(qs: np.ndarray, e: int) -> np.ndarray:
    byte, shift = k2_position(e)
    return (qs[:, byte].astype(np.int64) >> shift) & 3


def dequant_q2_k(blk: np.ndarray) -> np.ndarray:
    """[nb, 84] u8 -> [nb, 256] f64 (reading above)."""
    sc = blk[:, 0:16].astype(np.int64)
    qs = blk[:, 16:80]
    d, dmin = f16_field(blk[:, 80:82]), f16_field(blk[:, 82:84])
    out = np.empty((blk.shape[0], 256), dtype=np.float64)
    for e in range(256):
        j = e // 16
        out[:, e] = d * (sc[:, j] & 15) * q2_code(qs, e) - dmin * (sc[:, j] >> 4)
    return out


def q3k_scale6(s: np.ndarray, i: int) -> np.ndarray:
    """Sub-block scale i (0..15, unsigned 6 bits) of a Q3_K block from its 12
    scale bytes s [nb, 12] (reading: GGUF packing): the low 4 bits are the low
    (i < 8) or high (i >= 8) nibble of byte i % 8, the top 2 bits are bits
    2 * (i // 4) .. +1 of byte 8 + i % 4."""
    s = s.astype(np.int64)
    low = (s[:, i % 8] & 15) if i < 8 else (s[:, i % 8] >> 4)
    top = (s[:, 8 + i % 4] >> (2 * (i // 4))) & 3
    return low | (top << 4)


def q3_code(hmask: np.ndarray, qs: np.ndarray, e: int) -> np.ndarray:
    """Signed 3-bit code (-4..3) of element e: its 2-bit code, less 4 when bit
    e // 32 of hmask[e % 32] is clear."""
    hbit = (hmask[:, e % 32].astype(np.int64) >> (e // 32)) & 1
    return q2_code(qs, e) - 4 * (1 - hbit)


def dequant_q3_k(blk: np.ndarray) -> np.ndarray:
    """[nb, 110] u8 -> [nb, 256] f64 (reading above)."""
    hmask, qs, s = blk[:, 0:32], blk[:, 32:96], blk[:, 96:108]
    d = f16_field(blk[:, 108:110])
    out = np.empty((blk.shape[0], 256), dtype=np.float64)
    for e in range(256):
        out[:, e] = d * (q3k_scale6(s, e // 16) - 32) * q3_code(hmask, qs, e)
    return out


_DECODERS = {Q4_0: dequant_q4_0, Q4_1: dequant_q4_1, Q5_0: dequant_q5_0, Q5_1: dequant_q5_1,
             Q2_K: dequant_q2_k, Q3_K: dequant_q3_k,
             Q8_0: dequant_q8_0, Q4_K: dequant_q4_k, Q5_K: dequant_q5_k, Q6_K: dequant_q6_k}


def dequant(w: np.ndarray, qtype: int, N: int, K: int) -> np.ndarray:
    """Weight tensor [N, K/blk * block_bytes] u8 ([ov39119] "Why a new primitive")
    -> decoded weights [N, K] f64.  Blocks run along K within a row."""
    bv, bb = BLOCK_VALUES[qtype], BLOCK_BYTES[qtype]
    blk = np.ascontiguousarray(w, dtype=np.uint8).reshape(N * (K // bv), bb)
    return _DECODERS[qtype](blk).reshape(N, K)


# ----------------------------------------------------------------------------
# Q6_K plane regrouping ([ov39119] Transformation: QL[nblk][128] | QH[nblk][64]
# | SC[nblk][16] | D[nblk]; same size and contents)
# ----------------------------------------------------------------------------

def q6k_planes_offsets(nblk: int):
    """Byte offsets of QL, QH, SC, D and the total size."""
    return 0, 128 * nblk, 192 * nblk, 208 * nblk, 210 * nblk


def q6k_to_planes(w: np.ndarray) -> np.ndarray:
    """Raw Q6_K bytes (any shape, whole blocks in row-major block order) -> planes."""
    blk = np.ascontiguousarray(w, dtype=np.uint8).reshape(-1, 210)
    return np.concatenate([blk[:, 0:128].ravel(), blk[:, 128:192].ravel(),
                           blk[:, 192:208].ravel(), blk[:, 208:210].ravel()])


def q6k_from_planes(p: np.ndarray, nblk: int) -> np.ndarray:
    """Planes -> raw Q6_K blocks [nblk, 210]."""
    o_ql, o_qh, o_sc, o_d, total = q6k_planes_offsets(nblk)
    p = np.asarray(p, dtype=np.uint8)
    assert p.size == total
    blk = np.empty((nblk, 210), dtype=np.uint8)
    blk[:, 0:128] = p[o_ql:o_qh].reshape(nblk, 128)
    blk[:, 128:192] = p[o_qh:o_sc].reshape(nblk, 64)
    blk[:, 192:208] = p[o_sc:o_d].reshape(nblk, 16)
    blk[:, 208:210] = p[o_d:total].reshape(nblk, 2)
    return blk


def dequant_q6k_planes(p: np.ndarray, N: int, K: int) -> np.ndarray:
    """Decode straight from the plane layout: block b = n*(K/256) + kb reads
    QL[b], QH[b], SC[b], D[b]."""
    nblk = N * K // 256
    o_ql, o_qh, o_sc, o_d, total = q6k_planes_offsets(nblk)
    p = np.asarray(p, dtype=np.uint8)
    ql = p[o_ql:o_qh].reshape(nblk, 128)
    qh = p[o_qh:o_sc].reshape(nblk, 64)
    sc = p[o_sc:o_d].reshape(nblk, 16)
    d = f16_field(p[o_d:total].reshape(nblk, 2))
    return dequant_q6_k_fields(ql, qh, sc, d).reshape(N, K)


# ----------------------------------------------------------------------------
# exact matmul (the plain definition the fused GEMM and the decode-once arm reach
# up to rounding; [ov39119] Tests: expected values from the exact dequantization)
# ----------------------------------------------------------------------------

def matmul_exact(x: np.ndarray, w64: np.ndarray, residual: np.ndarray | None = None) -> np.ndarray:
    """ref[m, n] = sum_k x[m, k] * w[n, k] (+ residual[m, n]), all float64.
    ([ov39119]: MatMul(A, W, transpose_b=true); a following same-shape Add is fused.)"""
    ref = np.asarray(x, dtype=np.float64) @ np.asarray(w64, dtype=np.float64).T
    if residual is not None:
        ref = ref + np.asarray(residual, dtype=np.float64)
    return ref


# ----------------------------------------------------------------------------
# the int8 GEMV path, restated ([ov39119] Implementation: quantize activations per
# 32 values, int8 dot products directly against the blocks)
# ----------------------------------------------------------------------------

def quantize_act_q8(x32: np.ndarray):
    """Per-32 activation quantizer, all in f32 with IEEE rounding:
      amax = max |x| over the block
      d_a  = amax / 127
      id   = 1 / d_a   (0 when d_a == 0)
      qa   = round_half_away(clamp(x * id, -127, 127))
      s    = sum of qa over the block (int)
    x32: [M, K] float32 with K % 32 == 0.  Returns qa [M,K] int8, d_a [M,K/32]
    float32, s [M,K/32] int32.
    """
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    M, K = x32.shape
    xb = x32.reshape(M, K // 32, 32)
    amax = np.max(np.abs(xb), axis=2)
    d_a = (amax / np.float32(127.0)).astype(np.float32)
    with np.errstate(divide="ignore"):
        idv = np.where(d_a != 0, np.float32(1.0) / d_a, np.float32(0.0)).astype(np.float32)
    v = (xb * idv[:, :, None]).astype(np.float32)
    v = np.fmin(np.fmax(v, np.float32(-127.0)), np.float32(127.0))
    v64 = v.astype(np.float64)                     # exact; floor(|v| + 0.5) is exact in f64
    qa = (np.sign(v64) * np.floor(np.abs(v64) + 0.5)).astype(np.int8)
    s = qa.astype(np.int32).sum(axis=2).astype(np.int32)
    return qa.reshape(M, K), d_a, s


def weight_int_terms(w: np.ndarray, qtype: int, N: int, K: int):
    """Integer weight values q_w [N, K] (int64) and the per-sub-block factors.

    Returns (q_w, sub, scale, minv) where `sub` is the sub-block width (32, or
    16 for Q6_K), scale [N, K/sub] f64 multiplies the sub-block's integer dot and
    minv [N, K/sub] f64 (zero for Q8_0/Q6_K) multiplies d_a * s of its
    activation block, so that w = scale * q_w - minv element by element.
      Q4_0: q_w = q - 8,    scale = d;   Q5_0: q_w = q5 - 16, scale = d
      Q4_1: q_w = q,        scale = d, minv = -m;   Q5_1: q_w = q5, scale = d, minv = -m
      Q8_0: q_w = q,        scale = d
      Q4_K: q_w = nibble,   scale = d*sc_j, minv = dmin*m_j
      Q5_K: q_w = q5,       scale = d*sc_j, minv = dmin*m_j
      Q6_K: q_w = q6 - 32,  scale = d*scales[j] (16-wide sub-blocks)
      Q2_K: q_w = q2,       scale = d*(sc_j & 15), minv = dmin*(sc_j >> 4) (16-wide)
      Q3_K: q_w = q3,       scale = d*(scale6_j - 32) (16-wide)
    """
    bv, bb = BLOCK_VALUES[qtype], BLOCK_BYTES[qtype]
    nb = N * (K // bv)
    blk = np.ascontiguousarray(w, dtype=np.uint8).reshape(nb, bb)
    if qtype in (Q4_0, Q4_1, Q5_0, Q5_1):
        # Q4_0: q_w = q - 8, Q5_0: q_w = q5 - 16 (scale d); Q4_1 / Q5_1: q_w = q (or q5),
        # scale d, and the added min as minv = -m (w = scale * q_w - minv)
        q_off = {Q4_0: 2, Q4_1: 4, Q5_0: 6, Q5_1: 8}[qtype]
        qs = blk[:, q_off:q_off + 16]
        q = np.stack([b32_nibble(qs, e) for e in range(32)], axis=1)
        if qtype in (Q5_0, Q5_1):
            qh = blk[:, q_off - 4:q_off]
            q = q + 16 * np.stack([b32_fifth_bit(qh, e) for e in range(32)], axis=1)
        d = f16_field(blk[:, 0:2])
        if qtype in (Q4_0, Q5_0):
            q = q - (8 if qtype == Q4_0 else 16)
            minv = np.zeros(nb)
        else:
            minv = -f16_field(blk[:, 2:4])
        return q.reshape(N, K), 32, d.reshape(N, -1), minv.reshape(N, -1)
    if qtype == Q8_0:
        q = blk[:, 2:34].view(np.int8).astype(np.int64)
        scale = f16_field(blk[:, 0:2])[:, None]
        return q.reshape(N, K), 32, scale.reshape(N, -1), np.zeros((N, K // 32))
    if qtype in (Q4_K, Q5_K):
        d, dmin = f16_field(blk[:, 0:2]), f16_field(blk[:, 2:4])
        s = blk[:, 4:16]
        q = np.empty((nb, 256), dtype=np.int64)
        for e in range(256):
            if qtype == Q4_K:
                q[:, e] = q4k_nibble(blk[:, 16:144], e)
            else:
                hi = (blk[:, 16 + e % 32].astype(np.int64) >> (e // 32)) & 1
                q[:, e] = q4k_nibble(blk[:, 48:176], e) + 16 * hi
        scale = np.stack([d * decode_6bit(s, j) for j in range(8)], axis=1)
        minv = np.stack([dmin * decode_6bit(s, j + 8) for j in range(8)], axis=1)
        return q.reshape(N, K), 32, scale.reshape(N, -1), minv.reshape(N, -1)
    if qtype == Q2_K:
        sc = blk[:, 0:16].astype(np.int64)
        d, dmin = f16_field(blk[:, 80:82]), f16_field(blk[:, 82:84])
        q = np.stack([q2_code(blk[:, 16:80], e) for e in range(256)], axis=1)
        return q.reshape(N, K), 16, (d[:, None] * (sc & 15)).reshape(N, -1), (dmin[:, None] * (sc >> 4)).reshape(N, -1)
    if qtype == Q3_K:
        d = f16_field(blk[:, 108:110])
        q = np.stack([q3_code(blk[:, 0:32], blk[:, 32:96], e) for e in range(256)], axis=1)
        scale = np.stack([d * (q3k_scale6(blk[:, 96:108], j) - 32) for j in range(16)], axis=1)
        return q.reshape(N, K), 16, scale.reshape(N, -1), np.zeros((N, K // 16))
    if qtype == Q6_K:
        ql, qh = blk[:, 0:128], blk[:, 128:192]
        sc = blk[:, 192:208].view(np.int8).astype(np.float64)
        d = f16_field(blk[:, 208:210])
        q = np.stack([q6k_q6(ql, qh, e) - 32 for e in range(256)], axis=1)
        return q.reshape(N, K), 16, (d[:, None] * sc).reshape(N, -1), np.zeros((N, K // 16))
    raise ValueError(qtype)


def int8_dots(q_w: np.ndarray, sub: int, qa: np.ndarray) -> np.ndarray:
    """Integer sub-block dots D[m, n, j] = sum over sub-block j of q_w[n,k]*qa[m,k]."""
    N, K = q_w.shape
    M = qa.shape[0]
    qw3 = q_w.reshape(N, K // sub, sub)
    qa3 = qa.astype(np.int64).reshape(M, K // sub, sub)
    return np.einsum("njl,mjl->mnj", qw3, qa3)


def gemv_int8_path(w: np.ndarray, qtype: int, N: int, K: int, x32: np.ndarray,
                   residual: np.ndarray | None = None, return_terms: bool = False):
    """y[m, n] = sum_j scale[n,j] * d_a[m,b(j)] * D[m,n,j]
                - sum_j minv[n,j]  * d_a[m,b(j)] * s_j[m,j]   (+ residual)
    with b(j) the 32-wide activation block holding sub-block j (b = j for 32-wide
    sub-blocks, b = j // 2 for the 16-wide ones of Q2_K/Q3_K/Q6_K) and s_j the
    sum of the activation codes over sub-block j itself (the block's s for
    32-wide sub-blocks, one half of it for 16-wide ones).  Terms in float64."""
    qa, d_a, s = quantize_act_q8(x32)
    q_w, sub, scale, minv = weight_int_terms(w, qtype, N, K)
    D = int8_dots(q_w, sub, qa)                                # [M, N, K/sub] int64
    per = 32 // sub                                            # sub-blocks per activation block
    da_j = np.repeat(d_a.astype(np.float64), per, axis=1)      # [M, K/sub]
    M = qa.shape[0]
    s_j = qa.astype(np.int64).reshape(M, K // sub, sub).sum(axis=2).astype(np.float64)
    y = np.einsum("nj,mj,mnj->mn", scale, da_j, D.astype(np.float64))
    y = y - np.einsum("nj,mj,mj->mn", minv, da_j, s_j)
    if residual is not None:
        y = y + np.asarray(residual, dtype=np.float64)
    if return_terms:
        return y, dict(qa=qa, d_a=d_a, s=s, D=D)
    return y


# ----------------------------------------------------------------------------
# decode-once K-padded buffer ([rocm37] How it works / Correctness)
# ----------------------------------------------------------------------------

def dequant_padded_bits(w: np.ndarray, qtype: int, N: int, K: int, ld: int, odt: str) -> np.ndarray:
    """[N, ld] u16 bit patterns: out[n, k] = round(w[n, k]) to f16 or bf16 for
    k < K, and 0 in the pad columns K..ld-1."""
    w64 = dequant(w, qtype, N, K)
    out = np.zeros((N, ld), dtype=np.uint16)
    rnd = round_f64_to_f16_bits if odt == "f16" else round_f64_to_bf16_bits
    out[:, :K] = rnd(w64)
    return out


# ----------------------------------------------------------------------------
# MoE expert matmul ([ll28301] Overview: mul_mm_id)
# ----------------------------------------------------------------------------

def moe_mm_id_exact(w_experts, qtype: int, n_expert: int, N: int, K: int, x: np.ndarray,
                    ids: np.ndarray, residual: np.ndarray | None = None,
                    token_rows: np.ndarray | None = None) -> np.ndarray:
    """y[t, k, :] = x[t, :] . W_{ids[t, k]}^T (+ residual[t, k, :]), float64.
    x [T, K] (the same activation row for all of a token's slots) or [T, top_k, K]
    (one row per slot: y[t, k, :] = x[t, k, :] . W_{ids[t, k]}^T); ids [T, top_k].
    An id outside [0, n_expert) selects no expert: that row stays NaN (reading:
    the pages route every slot to a real expert; the library leaves such rows
    unwritten).  token_rows optionally restricts the evaluation to those tokens
    (NaN elsewhere)."""
    T, top_k = ids.shape
    rb = K // BLOCK_VALUES[qtype] * BLOCK_BYTES[qtype]
    wE = np.asarray(w_experts, dtype=np.uint8).reshape(n_expert, N, rb)
    x64 = np.asarray(x, dtype=np.float64)
    y = np.full((T, top_k, N), np.nan)
    rows = range(T) if token_rows is None else token_rows
    decoded = {}
    for t in rows:
        for k in range(top_k):
            e = int(ids[t, k])
            if not 0 <= e < n_expert:
                continue
            if e not in decoded:
                decoded[e] = dequant(wE[e], qtype, N, K)
            y[t, k] = decoded[e] @ (x64[t, k] if x64.ndim == 3 else x64[t])
    if residual is not None:
        y = y + np.asarray(residual, dtype=np.float64)
    return y


def moe_mv_id_int8(w_experts, qtype: int, n_expert: int, N: int, K: int, x32: np.ndarray,
                   ids: np.ndarray, residual: np.ndarray | None = None) -> np.ndarray:
    """The expert GEMM's decode form (mul_mv_id): every routed row (t, k) is
    the int8-path GEMV (gemv_int8_path, OpenVINO PR #39119 "Implementation",
    GEMV row) of its activation row -- x32[t] ([T, K]) or x32[t, k]
    ([T, top_k, K]) -- against expert ids[t, k].  Rows without a valid expert
    stay NaN, as in moe_mm_id_exact."""
    T, top_k = ids.shape
    rb = K // BLOCK_VALUES[qtype] * BLOCK_BYTES[qtype]
    wE = np.asarray(w_experts, dtype=np.uint8).reshape(n_expert, N, rb)
    x32 = np.asarray(x32, dtype=np.float32)
    y = np.full((T, top_k, N), np.nan)
    for t in range(T):
        for k in range(top_k):
            e = int(ids[t, k])
            if not 0 <= e < n_expert:
                continue
            row = x32[t, k] if x32.ndim == 3 else x32[t]
            r = None if residual is None else np.asarray(residual, dtype=np.float64)[t, k][None, :]
            y[t, k] = gemv_int8_path(wE[e], qtype, N, K, row[None, :], r)[0]
    return y


def moe_routing(ids: np.ndarray, n_expert: int):
    """Routing facts that any valid grouping must reproduce: per-expert row count
    and exclusive prefix offsets; rows of expert e are the (t, k) with ids == e.
    Ids outside [0, n_expert) select no expert and are not counted."""
    flat = np.asarray(ids).ravel()
    valid = flat[(flat >= 0) & (flat < n_expert)]
    counts = np.bincount(valid, minlength=n_expert).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)[:-1]])
    return counts, offsets
