// Per-element GGUF block decoders (device).  Block structs follow the GGUF
// on-disk layout (GGUF Support Proposal for mobius, section 7 "Quantization
// Format Deep Dive" and the 1.2 type table; OpenVINO PR #39119 "Transformation"
// for the Q6_K fields):
//   Q4_0  {d f16, qs[16]}                                    w = (q - 8)*d
//   Q4_1  {d, m f16, qs[16]}                                 w = q*d + m
//   Q5_0  {d f16, qh[4], qs[16]}                             w = (q5 - 16)*d
//   Q5_1  {d, m f16, qh[4], qs[16]}                          w = q5*d + m
//         (32 values; element e < 16 is the low nibble of qs[e], e >= 16 the
//         high nibble of qs[e - 16]; bit e of the little-endian qh word is the
//         fifth bit of element e)
//   Q8_0  {d f16, qs[32] i8}                                 w = d*q
//   Q4_K  {d, dmin f16, scales[12], qs[128]}                 w = d*sc_j*q - dmin*m_j
//   Q5_K  {d, dmin f16, scales[12], qh[32], qs[128]}         w = d*sc_j*q5 - dmin*m_j
//   Q6_K  {ql[128], qh[64], scales[16] i8, d f16}            w = d*scales[e/16]*(q6 - 32)
//   Q2_K  {scales[16], qs[64], d, dmin f16}                  w = d*(sc&15)*q2 - dmin*(sc>>4)
//   Q3_K  {hmask[32], qs[64], scales[12], d f16}             w = d*(scale6 - 32)*q3
//         (256 values, sub-block e/16; element 128h + 32j + 16p + l takes bits
//         2j..2j+1 of qs[32h + 16p + l]; Q3_K: q3 = q2 - 4 when bit e/32 of
//         hmask[e%32] is clear, scale6 i = low / high nibble of byte i%8 (i < 8 /
//         i >= 8) | bits 2(i/4)..+1 of byte 8 + i%4 << 4)
// The min is subtracted exactly, never folded into a rounded integer zero
// point (OpenVINO PR #38696, "Details").
#pragma once
#include "common.cuh"

namespace gg {

__host__ __device__ constexpr bool block32(int qt) {
    return qt == GGUF_Q4_0 || qt == GGUF_Q4_1 || qt == GGUF_Q5_0 || qt == GGUF_Q5_1 || qt == GGUF_Q8_0;
}
__host__ __device__ constexpr int block_values(int qt) { return block32(qt) ? 32 : 256; }
__host__ __device__ constexpr int block_bytes(int qt) {
    return qt == GGUF_Q4_0 ? 18 : qt == GGUF_Q4_1 ? 20 : qt == GGUF_Q5_0 ? 22 : qt == GGUF_Q5_1 ? 24
         : qt == GGUF_Q8_0 ? 34 : qt == GGUF_Q2_K ? 84 : qt == GGUF_Q3_K ? 110 : qt == GGUF_Q4_K ? 144
         : qt == GGUF_Q5_K ? 176 : 210;
}
// the 2- and 3-bit K-quants (16 sub-blocks of 16 values, 2-byte aligned blocks)
__host__ __device__ constexpr bool k23(int qt) { return qt == GGUF_Q2_K || qt == GGUF_Q3_K; }
// byte offset of the 16 code bytes inside a 32-value Q4/Q5 block (the qh word precedes them)
__host__ __device__ constexpr int b32_qs_offset(int qt) {
    return qt == GGUF_Q4_0 ? 2 : qt == GGUF_Q4_1 ? 4 : qt == GGUF_Q5_0 ? 6 : 8;
}
__host__ __device__ constexpr bool b32_has_min(int qt) { return qt == GGUF_Q4_1 || qt == GGUF_Q5_1; }
__host__ __device__ constexpr bool b32_has_qh(int qt) { return qt == GGUF_Q5_0 || qt == GGUF_Q5_1; }
// the implicit zero point of the symmetric formats
__host__ __device__ constexpr int b32_zero_point(int qt) { return qt == GGUF_Q4_0 ? 8 : qt == GGUF_Q5_0 ? 16 : 0; }

__device__ __forceinline__ float ld_f16_bytes(const uint8_t* p) {
    return f16_bits_to_float((uint32_t)p[0] | ((uint32_t)p[1] << 8));
}

// Sub-block scale (i < 8) or min (i >= 8) from the 12 packed bytes.
__device__ __forceinline__ int kquant_6bit(const uint8_t* s, int i) {
    const int j = i & 7, mn = i >> 3;
    if (j < 4) return s[j + 4 * mn] & 63;
    const int low = mn ? (s[j + 4] >> 4) : (s[j + 4] & 15);
    return low | ((s[j - 4 + 4 * mn] >> 6) << 4);
}

// 4-bit code of element e of a Q4_K/Q5_K super-block (qs = its 128 bytes).
__device__ __forceinline__ int kquant_nibble(const uint8_t* qs, int e) {
    const int p = e >> 6, r = e & 63;
    const int byte = qs[32 * p + (r & 31)];
    return r < 32 ? (byte & 15) : (byte >> 4);
}

// Q6_K code (0..63) of element e from its ql/qh fields.
__device__ __forceinline__ int q6k_code(const uint8_t* ql, const uint8_t* qh, int e) {
    const int h = e >> 7, r = e & 127, g = r >> 5, l = r & 31;
    const int b = ql[64 * h + 32 * (g & 1) + l];
    const int lo = g < 2 ? (b & 15) : (b >> 4);
    const int hi = (qh[32 * h + l] >> (2 * g)) & 3;
    return lo | (hi << 4);
}

// a - b for exact f32 operands, rounded to odd: toward zero, then the last
// bit set when the difference was not exact (Knuth's two-sum gives the exact
// error of the nearest-rounded difference).  A value rounded to odd in f32 and
// then to nearest in a type with at least two fewer significant bits (f16: 11,
// bf16: 8 against f32's 24) is the correctly rounded exact difference -- one
// rounding, not two.
__device__ __forceinline__ float sub_round_odd(float a, float b) {
    const float s = __fsub_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(-b, bb));
    const float t = __fsub_rz(a, b);
    return (err != 0.f && isfinite(t)) ? __uint_as_float(__float_as_uint(t) | 1u) : t;   // inf, NaN pass as they are
}

// 2-bit code of element e of a Q2_K / Q3_K super-block (qs = its 64 code bytes).
__device__ __forceinline__ int k2_code(const uint8_t* qs, int e) {
    const int h = e >> 7, j = (e >> 5) & 3;
    return (qs[32 * h + (e & 31)] >> (2 * j)) & 3;
}

// Unsigned 6-bit scale i (0..15) of a Q3_K block from its 12 scale bytes.
__device__ __forceinline__ int q3k_scale6(const uint8_t* s, int i) {
    const int low = i < 8 ? (s[i & 7] & 15) : (s[i & 7] >> 4);
    return low | (((s[8 + (i & 3)] >> (2 * (i >> 2))) & 3) << 4);
}

// Weight value of element e of one block as f32.  Every product is exact in
// f32 (d, dmin: 11 significant bits; sc, m: 6; q: at most 6); a K-quant's
// "- dmin*m" is rounded to odd (sub_round_odd), so that the one rounding to
// the output type is the correct rounding of the exact weight.
template <int QT>
__device__ __forceinline__ float decode_elem(const uint8_t* blk, int e) {
    if constexpr (QT == GGUF_Q4_0 || QT == GGUF_Q4_1 || QT == GGUF_Q5_0 || QT == GGUF_Q5_1) {
        const uint8_t* qs = blk + b32_qs_offset(QT);
        int q = (e < 16) ? (qs[e] & 15) : (qs[e - 16] >> 4);
        if (b32_has_qh(QT)) {
            const uint8_t* qh = qs - 4;
            q += 16 * ((qh[e >> 3] >> (e & 7)) & 1);
        }
        const float d = ld_f16_bytes(blk);
        // d*(q - zp) and q*d are exact in f32; q*d + m is rounded to odd, so the
        // one rounding to the output type is the correct rounding of the weight
        if (b32_has_min(QT)) return sub_round_odd(d * (float)q, -ld_f16_bytes(blk + 2));
        return d * (float)(q - b32_zero_point(QT));
    } else if (QT == GGUF_Q8_0) {
        return ld_f16_bytes(blk) * (float)static_cast<int8_t>(blk[2 + e]);
    } else if (QT == GGUF_Q4_K || QT == GGUF_Q5_K) {
        const float d = ld_f16_bytes(blk), dmin = ld_f16_bytes(blk + 2);
        const uint8_t* s = blk + 4;
        const int j = e >> 5;
        int q;
        if (QT == GGUF_Q4_K) {
            q = kquant_nibble(blk + 16, e);
        } else {
            q = kquant_nibble(blk + 48, e) + 16 * ((blk[16 + (e & 31)] >> j) & 1);
        }
        return sub_round_odd((d * (float)kquant_6bit(s, j)) * (float)q, dmin * (float)kquant_6bit(s, j + 8));
    } else if (QT == GGUF_Q2_K) {
        // d*sc*q2 (11 + 4 + 2 bits) and dmin*m are exact; the difference is rounded to odd
        const int sc = blk[e >> 4];
        const float d = ld_f16_bytes(blk + 80), dmin = ld_f16_bytes(blk + 82);
        return sub_round_odd((d * (float)(sc & 15)) * (float)k2_code(blk + 16, e), dmin * (float)(sc >> 4));
    } else if (QT == GGUF_Q3_K) {
        // d*(scale6 - 32)*q3: 11 + 6 + 3 significant bits, exact in f32
        const int q3 = k2_code(blk + 32, e) - 4 * (1 - ((blk[e & 31] >> (e >> 5)) & 1));
        return (ld_f16_bytes(blk + 108) * (float)(q3k_scale6(blk + 96, e >> 4) - 32)) * (float)q3;
    } else {
        const float d = ld_f16_bytes(blk + 208);
        const int8_t sc = static_cast<int8_t>(blk[192 + (e >> 4)]);
        return (d * (float)sc) * (float)(q6k_code(blk, blk + 128, e) - 32);
    }
}

// Q6_K element e of block b straight from the planes (nblk blocks in total).
__device__ __forceinline__ float decode_q6k_planes_elem(const uint8_t* planes, int64_t nblk, int64_t b, int e) {
    const uint8_t* ql = planes + 128 * b;
    const uint8_t* qh = planes + 128 * nblk + 64 * b;
    const int8_t sc = static_cast<int8_t>(planes[192 * nblk + 16 * b + (e >> 4)]);
    const float d = ld_f16_bytes(planes + 208 * nblk + 2 * b);
    return (d * (float)sc) * (float)(q6k_code(ql, qh, e) - 32);
}

}  // namespace gg
