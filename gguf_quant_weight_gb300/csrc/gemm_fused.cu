// Fused prefill GEMM on GGUF blocks: Y = X . W^T (+ residual) with the weight
// decoded inside the kernel.
//
// OpenVINO PR #39119 "FullyConnectedGGUF", "Implementation", DPAS prefill row:
// each 256-value weight block is decoded once into on-chip memory and reused
// across all the activation rows of the tile; block loading overlaps decoding;
// the tile grows with the row count.
//
// GB300 shape of it (one 128-weight-row x BN-token tile per CTA, swap-AB):
//   warp 0     TMA producer of the raw weights: the tile's super-block bytes
//              (one 256-value column of 128 rows per raw slot: Q4_K/Q5_K/Q8_0
//              blocks, raw Q6_K rows from their 16-byte boundary, or the four
//              Q6_K planes), up to RS super-blocks ahead -- its own warp, so the
//              weight stream never waits on the MMA's operand stages
//   warp 1     TMEM allocation and tcgen05.mma issue (128 x BN x 16 per MMA,
//              f32 accumulators in TMEM), one commit per stage; at BN <= 128
//              one more warp (after the decoders) issues too, half of every
//              k step's MMAs, into its own accumulator
//   warp 2     TMA producer of the f16 activation tile of each 64-value k step
//   warps 3..  decoders (16 warps for Q4_K/Q5_K/Q6_K planes, 8 otherwise):
//              each k step they turn 128 rows x 64 values of raw bytes into f16
//              (packed f16 math: w = fl16(d*sc)*q - fl16(dmin*m) in one fused
//              multiply-add per value pair; the scales of a super-block are
//              computed once, at its first k step), written into tensor
//              memory with tcgen05.st, where the MMA reads its A operand; then
//              the epilogue (TMEM -> registers, + residual, store)
// The MMA never waits on decode of the same stage it consumes: stages ring
// through S slots, so decode of step i+1.. overlaps the MMAs of step i.
// When the tiles would leave SMs idle, K is split across CTAs (all tiles, or
// only those of the last, partial round); the slices' partial tiles meet in the
// workspace and the last slice of a tile adds them in slice order.
#include <algorithm>
#include <cstdlib>
#include <cstring>

#include "tc_gemm.cuh"
#include "formats.cuh"

namespace gg {

namespace {

// decoder warps: 16 (each thread a quarter of a 64-value k step) for the
// layouts decoded from a per-super-block state, else 8 (each thread a half).
// Q4_K / Q5_K take 8 half-step warps below BN = 256: a warp's per-step work
// of waits, addresses and the TMEM store is then spread over twice the values
// (measured, Q5_K 14336 x 4096: M = 8 / 64 / 128 26.5 -> 24.2, 27.7 -> 25.8,
// 28.3 -> 27.1 us; MoE T = 32 / 512 43.3 -> 39.3, 73.8 -> 68.6 us), while the
// BN = 256 tiles of M >= 256 keep 16 (8 cost them 3-5 %).
__host__ __device__ constexpr bool state_decoder(int qt, int layout) {
    return qt == GGUF_Q4_K || qt == GGUF_Q5_K || (qt == GGUF_Q6_K && layout == GGUF_LAYOUT_Q6K_PLANES);
}
__host__ __device__ constexpr int decode_warps(int qt, int layout, int bn) {
    return state_decoder(qt, layout) && !((qt == GGUF_Q4_K || qt == GGUF_Q5_K) && bn <= 128) ? 16 : 8;
}
// MMA-issuing threads.  One tcgen05.mma costs the thread that issues it ~60
// cycles (more beside busy decoder warps) -- at BN <= 128 far longer than the
// tensor core takes to run it -- while threads in different warps issue in
// parallel (measured: 1, 2, 4 issuing warps of 128 x 16 x 16 MMAs give 1, 1.7
// and 3.5 times the rate).  So NI threads, one per warp, split the four MMAs
// of each k step, each accumulating into its own BN TMEM columns (K split
// NI ways); the epilogue adds the NI partial sums.  (Two, not four: the TMEM
// columns are worth more as operand stages.)
// Two CTAs per SM (CTAS = 2, each with half of tensor memory) take one issuer.
__host__ __device__ constexpr int mma_issuers(int bn, int ctas = 1) { return (bn <= 128 && ctas == 1) ? 2 : 1; }
// warp 0: raw-weight TMA producer; warp 1: TMEM + MMA issuer 0; warp 2:
// activation TMA producer; warps 3 .. 3+DW-1: decoders (and the epilogue);
// the last NI - 1 warps: MMA issuers 1 .. NI-1
__host__ __device__ constexpr int fused_threads(int qt, int layout, int bn, int ctas = 1) {
    return 96 + 32 * decode_warps(qt, layout, bn) + 32 * (mma_issuers(bn, ctas) - 1);
}

// bytes of one 256-value column of a weight row: eight 32-value blocks or one super-block
__host__ __device__ constexpr int col_bytes(int qt) { return block32(qt) ? 8 * block_bytes(qt) : block_bytes(qt); }
__host__ __device__ constexpr int raw_pitch(int qt, int layout) {
    // bytes per weight row in one raw slot (= the TMA box's inner extent): the
    // column, plus up to 14 leading bytes where it is boxed from a 16-byte
    // boundary (the 2-byte aligned super-blocks of raw Q6_K, Q2_K, Q3_K),
    // rounded up to an ODD multiple of 16 bytes: the decoder warps read 32
    // consecutive rows at once, and an even multiple puts them in a few banks
    // (a 128-byte pitch: every row in the same bank -- Q3_K ran 326 us at
    // 14336 x 4096, M <= 16, against 45 us for Q2_K)
    return (qt == GGUF_Q6_K && layout) ? 0
         : ((((col_bytes(qt) + (col_bytes(qt) % 16 ? 14 : 0) + 15) / 16) % 2 == 0)
                ? (col_bytes(qt) + (col_bytes(qt) % 16 ? 14 : 0) + 15) / 16 * 16 + 16
                : (col_bytes(qt) + (col_bytes(qt) % 16 ? 14 : 0) + 15) / 16 * 16);
}
static_assert(raw_pitch(GGUF_Q2_K, 0) == 112 && raw_pitch(GGUF_Q3_K, 0) == 144 && raw_pitch(GGUF_Q6_K, 0) == 240 &&
                  raw_pitch(GGUF_Q4_K, 0) == 144 && raw_pitch(GGUF_Q5_K, 0) == 176 && raw_pitch(GGUF_Q5_1, 0) == 208 &&
                  raw_pitch(GGUF_Q8_0, 0) == 272 && raw_pitch(GGUF_Q4_1, 0) == 176,
              "odd multiples of 16 bytes");
// bytes of one raw slot (128 rows); the Q6_K planes slot is QL | QH | SC | D
__host__ __device__ constexpr int raw_slot_bytes(int qt, int layout) {
    return (qt == GGUF_Q6_K && layout) ? 128 * (128 + 64 + 16 + 16) : 128 * raw_pitch(qt, layout);
}

// CTAS: CTAs resident per SM.  With two, each holds half of tensor memory
// (256 columns) and half of shared memory, so that one CTA's start-up,
// epilogue and decoder chain overlap the other's (the decoder-bound tiles:
// MoE work items with few token columns).
template <int BN, int RAW, int CTAS = 1>
struct FusedCfg {
    // The decoded weight tile (the MMA's A operand, 128 rows x 64 f16 per k
    // step) lives in tensor memory: decoders write it with tcgen05.st and the
    // MMA reads it from there, so shared memory carries only the activation
    // tiles (B) and the raw blocks.  One ring of S stages covers both operands
    // of a k step (one "full" barrier: the decoder warps plus the activation
    // TMA; one "empty" barrier: one commit per issuer), which keeps the
    // MMA-issuing threads' work per step small.
    static constexpr int NI = mma_issuers(BN, CTAS); // issuers; accumulator j at columns [j*BN, (j+1)*BN)
    static constexpr int A_COLS = 32;                 // TMEM columns per decoded stage
    static constexpr int A_COL0 = NI * BN < 32 ? 32 : NI * BN;   // first decoded-stage column
    static constexpr int B_BYTES = BN * 64 * 2;
    static constexpr int TMEM_COLS = 512 / CTAS;      // accumulators [0, NI*BN) + decoded stages
    // dynamic shared memory one CTA may use: all of it, or half of the SM's
    // 228 KB less the per-CTA reserve and the static scale array
    static constexpr int SMEM_CAP = CTAS == 1 ? 232448 : (233472 - 2 * 1024) / 2 - 4 * BN;
    // Stages: as many as tensor memory holds (up to 12) while shared memory
    // keeps three raw slots -- the activation tile of a step is requested
    // when its stage frees, and under the weight stream it lands ~3000 cycles
    // later, so the ring must reach that far ahead of the MMAs.  BN = 256
    // keeps four (its tiles are wide enough that the MMAs cover the wait).
    static constexpr int S_TMEM = (TMEM_COLS - A_COL0) / A_COLS;
    static constexpr int S_SMEM = (SMEM_CAP - 2048 - (CTAS == 1 ? 3 : 2) * RAW) / B_BYTES;
    static constexpr int S_MIN = S_TMEM < S_SMEM ? S_TMEM : S_SMEM;
    static constexpr int S = BN >= 256 ? 4 : (S_MIN > 12 ? 12 : S_MIN);
    // raw slots: what the activation stages leave (each covers four k steps)
    static constexpr int RS_FIT = (SMEM_CAP - 2048 - S * B_BYTES) / RAW;
    static constexpr int RS = RS_FIT > 6 ? 6 : RS_FIT;
    static constexpr int SMEM = S * B_BYTES + RS * RAW + 1024 + 512;   // + alignment + barriers
    static_assert(8 * (2 * S + 2 * RS + 2) + 8 <= 512, "barrier area");
    // usable: two raw slots at least (a configuration without them is only
    // ever inspected, never launched: the kernel asserts OK)
    static constexpr bool OK = RS >= 2 && S >= 2;
    static_assert(A_COL0 + S * A_COLS <= TMEM_COLS && NI * BN <= A_COL0 && 4 % NI == 0, "TMEM columns");
};

struct FusedParams {
    int64_t N, M;
    int KB;              // super-blocks along K
    const void* residual;
    void* y;
    int ydt;
    int* status;
    // grouped (MoE) mode: one CTA row per (expert, token tile) work item
    const int4* tiles;   // {expert, first row inside the expert's group, rows, 0}
    const int* ntiles;   // number of work items
    const int* offsets;  // [n_expert + 1] start of each expert's group in the gathered activations
    const int* rows;     // entry (token * top_k + slot) of every gathered row
    int full_width;      // measurement aid: MMAs always BN wide (no tile-skip)
    // split K (dense mode): grid z = ks slices of the super-blocks; every slice
    // writes its partial tile, the last to finish a tile adds them up
    int ks;
    float* partial;      // [tile][ks][BN][128] f32
    int* tickets;        // [tile], zero at launch
    // split form's tiles in launch order (1-D grid): the first n_full whole,
    // then every further tile as ks consecutive K slices
    int n_full, ntile_n;
    // power-of-two scale of each activation row's f16 copy (dense: row t0 +
    // col; grouped: gathered row gstart + col); the epilogue multiplies by it
    const float* xscale;
    // launched as a programmatic dependent of the activation conversion: the
    // weight stream and decoding start at once, what reads the conversion's
    // outputs waits for it (host-side launch choice)
    int pdl;
};

// barrier `id` over the first `threads` threads that reach it (whole warps)
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ uint4 lds128u(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds16u(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds_w2(uint32_t a) {   // 32-bit word at a 2-byte aligned address
    return lds16u(a) | (lds16u(a + 2) << 16);
}
__device__ __forceinline__ uint32_t byte_of(uint32_t w, int i) { return (w >> (8 * i)) & 0xFFu; }
__device__ __forceinline__ uint32_t word_of(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// ---- packed f16 decode
// A code byte b (0..255) becomes the f16 value 1024 + b by placing it under the
// exponent byte 0x64 (one byte permute makes two such values); subtracting
// 1024 (plus any bias) is exact, and one fused multiply-add applies the
// block's scale and min:  w = fl16(scale) * q - fl16(offset), rounded once.
__device__ __forceinline__ __half2 h2_bits(uint32_t v) { return *reinterpret_cast<const __half2*>(&v); }
__device__ __forceinline__ uint32_t bits_h2(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }

// codes of bytes 0,1 (lo) and 2,3 (hi) of w as f16 (1024 + b)
__device__ __forceinline__ __half2 magic_lo(uint32_t w) { return h2_bits(__byte_perm(w, 0x64646464u, 0x4140)); }
__device__ __forceinline__ __half2 magic_hi(uint32_t w) { return h2_bits(__byte_perm(w, 0x64646464u, 0x4342)); }

// 8 words of 4 codes (32 values) -> 4 chunks of 8 f16:  w = scale * (code - bias) - offset
// (scale2/offset2: per-16-value halves given separately for Q6_K's sub-blocks)
__device__ __forceinline__ void emit32_h(const uint32_t q4[8], __half2 bias, __half2 sc_a, __half2 off_a,
                                         __half2 sc_b, __half2 off_b, uint4 out[4]) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const __half2 sc = c < 2 ? sc_a : sc_b, off = c < 2 ? off_a : off_b;
        uint32_t h[4];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t w = q4[2 * c + t];
            h[2 * t] = bits_h2(__hfma2(__hsub2(magic_lo(w), bias), sc, __hneg2(off)));
            h[2 * t + 1] = bits_h2(__hfma2(__hsub2(magic_hi(w), bias), sc, __hneg2(off)));
        }
        out[c] = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// ---- per-super-block decoder state
// A decoder thread owns one weight row r and one half hf of every 64-value k
// step, i.e. the 32-value sub-blocks j = 2q + hf (q = 0..3) of each super-block
// (Q4_K/Q5_K) or the 16-value sub-blocks 8(q/2) + 2g, +1 with g = 2(q%2) + hf
// (Q6_K).  Everything that depends only on the super-block -- the f16 scale
// and min of those sub-blocks, Q5_K's high-bit bytes -- is read and computed
// once per super-block, leaving four lean k steps.
template <int QT, int LAYOUT>
struct KbState {
    __half2 sc[4], noff[4];   // per k step (Q6_K: first / second 16-value half)
    uint32_t qh[8];           // Q5_K: the 32 high-bit bytes
    // hh >= 0: a quarter-step decoder (16 warps) -- only its own 16 qh bytes
    // are kept (in qh[0..3]) and, for Q6_K, only its 16-value sub-block's scale
    // (in sc[q]); hh < 0: a half-step decoder
    __device__ __forceinline__ void prepare(uint32_t row, uint32_t slot, int r, int hf, int kb, int hh = -1) {
        if constexpr (QT == GGUF_Q4_K || QT == GGUF_Q5_K) {
            const uint4 hdr = lds128u(row);
            const float d = f16_bits_to_float(hdr.x), dmin = f16_bits_to_float(hdr.x >> 16);
            // 6-bit scale/min of sub-blocks 0..3 (low bytes) and 4..7 (packed)
            const uint32_t sc_lo = hdr.y & 0x3F3F3F3Fu, mn_lo = hdr.z & 0x3F3F3F3Fu;
            const uint32_t sc_hi = (hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u);
            const uint32_t mn_hi = ((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int j = 2 * q + hf;   // runtime only through hf
                const uint32_t scw = q < 2 ? sc_lo : sc_hi, mnw = q < 2 ? mn_lo : mn_hi;
                const int bi = (2 * q + hf) & 3;
                (void)j;
                sc[q] = __float2half2_rn(d * (float)byte_of(scw, bi));
                noff[q] = __hneg2(__float2half2_rn(dmin * (float)byte_of(mnw, bi)));
            }
            if constexpr (QT == GGUF_Q5_K) {
                if (hh >= 0) {
                    const uint4 h0 = lds128u(row + 16 + 16 * hh);
                    qh[0] = h0.x; qh[1] = h0.y; qh[2] = h0.z; qh[3] = h0.w;
                } else {
                    const uint4 h0 = lds128u(row + 16), h1 = lds128u(row + 32);
                    qh[0] = h0.x; qh[1] = h0.y; qh[2] = h0.z; qh[3] = h0.w;
                    qh[4] = h1.x; qh[5] = h1.y; qh[6] = h1.z; qh[7] = h1.w;
                }
            }
        } else if constexpr (QT == GGUF_Q6_K && LAYOUT == GGUF_LAYOUT_Q6K_PLANES) {
            const uint32_t sc_addr = slot + 128u * 192 + 16u * r;
            const uint32_t dq = slot + 128u * 208 + 16u * r + (uint32_t)((2 * kb) & 15);
            const float d = f16_bits_to_float(lds16u(dq));
            const uint4 scv = lds128u(sc_addr);   // the 16 signed scales
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int h = q >> 1;
                const int j0 = 8 * h + 4 * (q & 1) + 2 * hf;   // 8h + 2g
                const uint32_t w = word_of(scv, j0 >> 2);
                const int b = j0 & 3;
                if (hh >= 0) {
                    sc[q] = __float2half2_rn(d * (float)(int8_t)byte_of(w, b + hh));
                } else {
                    sc[q] = __float2half2_rn(d * (float)(int8_t)byte_of(w, b));
                    noff[q] = __float2half2_rn(d * (float)(int8_t)byte_of(w, b + 1));   // second half's scale
                }
            }
        }
    }
};

// A quarter of k step q of a super-block from a prepared state (Q4_K, Q5_K,
// Q6_K planes): values 32hf + 16hh .. +15 of the step (one 16-byte piece of the
// code bytes; Q6_K: exactly one 16-value sub-block).  HALF: the state was
// prepared for a half-step decoder (all of its 32 Q5_K high-bit bytes kept;
// Q4_K / Q5_K only).
template <int QT, int LAYOUT, bool HALF = false>
__device__ __forceinline__ void decode_quarter(const KbState<QT, LAYOUT>& st, uint32_t row, uint32_t slot, int r,
                                               int q, int hf, int hh, uint4 out[2]) {
    static_assert(!HALF || QT == GGUF_Q4_K || QT == GGUF_Q5_K, "half-step states: Q4_K / Q5_K");
    uint32_t q4[4];
    __half2 scv, noffv, bias;
    if constexpr (QT == GGUF_Q4_K || QT == GGUF_Q5_K) {
        const uint4 a = lds128u(row + (QT == GGUF_Q5_K ? 48 : 16) + 32 * q + 16 * hh);
        const uint32_t sh = 4u * (uint32_t)hf;
        const uint32_t rot = (uint32_t)(4 - (2 * q + hf)) & 31u;   // bit j of a byte -> bit 4
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t v = (word_of(a, i) >> sh) & 0x0F0F0F0Fu;
            if constexpr (QT == GGUF_Q5_K) {
                const uint32_t h = st.qh[(HALF ? 4 * hh : 0) + i];
                v |= __funnelshift_l(h, h, rot) & 0x10101010u;
            }
            q4[i] = v;
        }
        scv = st.sc[q];
        noffv = st.noff[q];
        bias = __float2half2_rn(1024.f);
    } else {
        const int h = q >> 1, g = 2 * (q & 1) + hf;
        // QL rows: 128-byte swizzle (16-byte chunk c of row r at c ^ (r % 8));
        // QH rows: 64-byte swizzle (chunk c of row r at c ^ ((r / 2) % 4))
        const uint32_t xc = (uint32_t)(4 * h + 2 * (g & 1) + hh) ^ (uint32_t)(r & 7);
        const uint32_t yc = (uint32_t)(2 * h + hh) ^ (uint32_t)((r >> 1) & 3);
        const uint4 x = lds128u(slot + 128u * r + (xc << 4));
        const uint4 y = lds128u(slot + 128u * 128 + 64u * r + (yc << 4));
        const uint32_t lsh = g < 2 ? 0u : 4u, hsh = 2u * (uint32_t)g;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            q4[i] = ((word_of(x, i) >> lsh) & 0x0F0F0F0Fu) | (((word_of(y, i) >> hsh) << 4) & 0x30303030u);
        scv = st.sc[q];   // this quarter's 16-value sub-block scale
        noffv = __float2half2_rn(0.f);
        bias = __float2half2_rn(1056.f);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint32_t h[4];
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const uint32_t w = q4[2 * c + t];
            h[2 * t] = bits_h2(__hfma2(__hsub2(magic_lo(w), bias), scv, noffv));
            h[2 * t + 1] = bits_h2(__hfma2(__hsub2(magic_hi(w), bias), scv, noffv));
        }
        out[c] = make_uint4(h[0], h[1], h[2], h[3]);
    }
}

// Q8_0 block J (0..7) of a 272-byte raw row: its f16 scale bits and its 32
// codes as 8 words.  The 34-byte blocks sit at 2-byte alignment, so the row is
// read as three aligned 16-byte pieces and the words are cut out with funnel
// shifts: with rows 272 = 17 x 16 bytes apart, 16-byte reads of 32 rows are
// free of bank conflicts (2-byte reads hit 8 distinct banks: 4-way).
template <int J>
__device__ __forceinline__ void q8_block(uint32_t row, uint32_t& d_bits, uint32_t q4[8]) {
    constexpr int B = (34 * J) & ~15, S = (34 * J) & 15, T = S + 2;   // piece start, scale and code offsets
    const uint4 c0 = lds128u(row + B), c1 = lds128u(row + B + 16), c2 = lds128u(row + B + 32);
    const uint32_t w[12] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w, c2.x, c2.y, c2.z, c2.w};
    d_bits = (S & 2) ? (w[S / 4] >> 16) : (w[S / 4] & 0xFFFFu);
#pragma unroll
    for (int i = 0; i < 8; ++i) q4[i] = (T & 2) ? __funnelshift_r(w[T / 4 + i], w[T / 4 + i + 1], 16) : w[T / 4 + i];
}

// Block J (0..7) of a raw row of eight 32-value Q4_0 / Q4_1 / Q5_0 / Q5_1
// blocks (8 * BB bytes, a multiple of 16): the f16 bits of d (and m), and the
// 32 codes as 8 words in element order (low nibbles of the 16 code bytes for
// elements 0..15, high nibbles for 16..31, the fifth bit from qh at bit 4).
// The blocks sit at 2-byte alignment: the 16-byte pieces covering the block
// (never past the row's end) are read and words cut out with funnel shifts.
template <int QT, int J>
__device__ __forceinline__ void b32_block(uint32_t row, uint32_t& d_bits, uint32_t& m_bits, uint32_t q4[8]) {
    constexpr int BB = block_bytes(QT), S0 = BB * J, B = S0 & ~15, NP = (S0 + BB - B + 15) / 16;
    static_assert(NP <= 3 && B + 16 * NP <= 8 * BB, "pieces stay inside the row");
    uint32_t w[12];
#pragma unroll
    for (int k = 0; k < NP; ++k) {
        const uint4 c = lds128u(row + B + 16 * k);
        w[4 * k] = c.x; w[4 * k + 1] = c.y; w[4 * k + 2] = c.z; w[4 * k + 3] = c.w;
    }
    auto half_at = [&](int off) -> uint32_t {   // 16 bits at byte S0 + off
        const int a = S0 + off - B;
        return (a & 2) ? (w[a / 4] >> 16) : (w[a / 4] & 0xFFFFu);
    };
    auto word_at = [&](int off) -> uint32_t {   // 32 bits at byte S0 + off (2-byte aligned)
        const int a = S0 + off - B;
        return (a & 2) ? __funnelshift_r(w[a / 4], w[a / 4 + 1], 16) : w[a / 4];
    };
    d_bits = half_at(0);
    m_bits = b32_has_min(QT) ? half_at(2) : 0u;
    constexpr int QO = b32_qs_offset(QT);
    uint32_t qh = 0;
    if constexpr (b32_has_qh(QT)) qh = word_at(QO - 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t q = word_at(QO + 4 * i);
        q4[i] = q & 0x0F0F0F0Fu;
        q4[4 + i] = (q >> 4) & 0x0F0F0F0Fu;
        if constexpr (b32_has_qh(QT)) {
            q4[i] |= (((qh >> (4 * i)) & 0xFu) * 0x00204081u & 0x01010101u) << 4;
            q4[4 + i] |= (((qh >> (16 + 4 * i)) & 0xFu) * 0x00204081u & 0x01010101u) << 4;
        }
    }
}

// Decode values 32*hf .. 32*hf+31 of k step q (values 64q .. 64q+63 of the
// super-block) of one weight row whose raw bytes start at shared address `row`.
template <int QT, int LAYOUT>
__device__ __forceinline__ void decode32(uint32_t row, uint32_t slot, int r, int q, int hf, int kb, uint4 out[4]) {
    static_assert(block32(QT) || k23(QT) || (QT == GGUF_Q6_K && LAYOUT == GGUF_LAYOUT_BLOCKS),
                  "the other layouts decode from a per-super-block state");
    (void)slot; (void)r; (void)kb;
    const __half2 zero2 = __float2half2_rn(0.f);
    if constexpr (QT == GGUF_Q8_0) {
        // signed codes: flipping the sign bit gives b = q + 128 in 0..255
        uint32_t db, q4[8];
        switch (2 * q + hf) {
            case 0: q8_block<0>(row, db, q4); break;
            case 1: q8_block<1>(row, db, q4); break;
            case 2: q8_block<2>(row, db, q4); break;
            case 3: q8_block<3>(row, db, q4); break;
            case 4: q8_block<4>(row, db, q4); break;
            case 5: q8_block<5>(row, db, q4); break;
            case 6: q8_block<6>(row, db, q4); break;
            default: q8_block<7>(row, db, q4); break;
        }
        const __half2 d2 = h2_bits(db * 0x10001u);
#pragma unroll
        for (int i = 0; i < 8; ++i) q4[i] ^= 0x80808080u;
        emit32_h(q4, __float2half2_rn(1152.f), d2, zero2, d2, zero2, out);
    } else if constexpr (block32(QT)) {
        // codes 0..15 (0..31 with the fifth bit): w = (q - zp) * d, or q * d + m
        // (one fused multiply-add, one rounding of the exact value)
        uint32_t db, mb, q4[8];
        switch (2 * q + hf) {
            case 0: b32_block<QT, 0>(row, db, mb, q4); break;
            case 1: b32_block<QT, 1>(row, db, mb, q4); break;
            case 2: b32_block<QT, 2>(row, db, mb, q4); break;
            case 3: b32_block<QT, 3>(row, db, mb, q4); break;
            case 4: b32_block<QT, 4>(row, db, mb, q4); break;
            case 5: b32_block<QT, 5>(row, db, mb, q4); break;
            case 6: b32_block<QT, 6>(row, db, mb, q4); break;
            default: b32_block<QT, 7>(row, db, mb, q4); break;
        }
        const __half2 d2 = h2_bits(db * 0x10001u);
        const __half2 noff = b32_has_min(QT) ? __hneg2(h2_bits(mb * 0x10001u)) : zero2;   // emit subtracts the offset
        emit32_h(q4, __float2half2_rn(1024.f + (float)b32_zero_point(QT)), d2, noff, d2, noff, out);
    } else if constexpr (k23(QT)) {
        // Q2_K / Q3_K: values 64q + 32hf + t = 128h + 32j + t with h = q/2,
        // j = 2(q%2) + hf; value t is bits 2j..2j+1 of qs[32h + t], in
        // sub-block 8h + 2j + t/16 (two 16-value halves, two scales)
        const int h = q >> 1, j = 2 * (q & 1) + hf, s0 = 8 * h + 2 * j;
        constexpr uint32_t QS = QT == GGUF_Q2_K ? 16 : 32;
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = (lds_w2(row + QS + 32u * h + 4u * i) >> (2 * j)) & 0x03030303u;
        if constexpr (QT == GGUF_Q2_K) {
            // w = fl16(d*sc) * q2 - fl16(dmin*m) per half
            const float d = f16_bits_to_float(lds16u(row + 80)), dmin = f16_bits_to_float(lds16u(row + 82));
            const uint32_t sw = lds16u(row + (uint32_t)s0);   // scale bytes s0, s0 + 1
            const float sa = (float)(sw & 15), ma = (float)((sw >> 4) & 15);
            const float sb = (float)((sw >> 8) & 15), mb = (float)((sw >> 12) & 15);
            emit32_h(c, __float2half2_rn(1024.f), __float2half2_rn(d * sa), __float2half2_rn(dmin * ma),
                     __float2half2_rn(d * sb), __float2half2_rn(dmin * mb), out);
        } else {
            // the high bit (bit 4h + j of hmask[t]) makes the code q3 + 4 (0..7)
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] |= ((lds_w2(row + 4u * i) >> (4 * h + j)) & 0x01010101u) << 2;
            const float d = f16_bits_to_float(lds16u(row + 108));
            const uint32_t lo = (s0 & 7) < 4 ? lds_w2(row + 96) : lds_w2(row + 100);   // bytes s0 % 8, s0 % 8 + 1
            const uint32_t w8 = lds_w2(row + 104);
            auto scale6 = [&](int i) {   // i = 8h + t with t = s0 % 8 or s0 % 8 + 1
                const uint32_t byte = (lo >> (8 * ((i & 7) & 3))) & 0xFF;
                const uint32_t low = i < 8 ? (byte & 15) : (byte >> 4);
                return (int)(low | ((((w8 >> (8 * (i & 3))) >> (2 * (i >> 2))) & 3) << 4)) - 32;
            };
            emit32_h(c, __float2half2_rn(1028.f), __float2half2_rn(d * (float)scale6(s0)), zero2,
                     __float2half2_rn(d * (float)scale6(s0 + 1)), zero2, out);
        }
    } else {
        // raw Q6_K: values 64q + 32hf + l = 128h + 32g + l with h = q/2, g = 2(q%2) + hf
        const int h = q >> 1, g = 2 * (q & 1) + hf;
        const uint32_t ql = row, qh = row + 128, sc = row + 192, dq = row + 208;   // 2-byte aligned
        const float d = f16_bits_to_float(lds16u(dq));
        uint32_t q4[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t x = lds_w2(ql + 64 * h + 32 * (g & 1) + 4 * i), y = lds_w2(qh + 32 * h + 4 * i);
            const uint32_t lo = g < 2 ? (x & 0x0F0F0F0Fu) : ((x >> 4) & 0x0F0F0F0Fu);
            q4[i] = lo | (((y >> (2 * g)) & 0x03030303u) << 4);
        }
        // two 16-value sub-blocks with signed scales: w = d*sc*(q6 - 32)
        const int j0 = 8 * h + 2 * g;
        const uint32_t scw = lds_w2(sc + (j0 & ~3));
        const __half2 s0 = __float2half2_rn(d * (float)(int8_t)byte_of(scw, j0 & 3));
        const __half2 s1 = __float2half2_rn(d * (float)(int8_t)byte_of(scw, (j0 & 3) + 1));
        emit32_h(q4, __float2half2_rn(1056.f), s0, zero2, s1, zero2, out);
    }
}

// SPLIT: the K-split form (a separate instantiation: its epilogue code in the
// kernel slowed the unsplit form by ~3 %, measured)
template <int QT, int LAYOUT, int BN, bool MOE, bool SPLIT, int CTAS = 1>
__global__ void __launch_bounds__(fused_threads(QT, LAYOUT, BN, CTAS), CTAS)
    fused_tc_kernel(const __grid_constant__ CUtensorMap tmW0, const __grid_constant__ CUtensorMap tmW1,
                    const __grid_constant__ CUtensorMap tmW2, const __grid_constant__ CUtensorMap tmW3,
                    const __grid_constant__ CUtensorMap tmB, const FusedParams fp) {
    constexpr int RAW = raw_slot_bytes(QT, LAYOUT);
    using C = FusedCfg<BN, RAW, CTAS>;
    static_assert(C::OK, "raw ring needs two slots");
    constexpr bool PLANES = QT == GGUF_Q6_K && LAYOUT == GGUF_LAYOUT_Q6K_PLANES;
    constexpr int PITCH = raw_pitch(QT, LAYOUT);
    constexpr int DW = decode_warps(QT, LAYOUT, BN);   // decoder warps
    constexpr int NI = C::NI;                      // MMA issuers
    // k steps a decoder warp takes per round: two for Q6_K (measured: raw
    // blocks 170 -> 101 us, planes 187 -> 182 us at M = 512 / 2048), one for
    // the others (two cost Q8_0 8 % at M = 4096 and Q5_K 7 % at M = 64)
    constexpr int DB = QT == GGUF_Q6_K ? 2 : 1;
    static_assert(4 % DB == 0 && DB <= C::S, "decode rounds");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = align_up_1024(smem_raw);
    uint8_t* sB = base;
    uint8_t* sR = sB + C::S * C::B_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sR + C::RS * RAW);    // decoded tile + activation tile ready
    uint64_t* empty = full + C::S;                                      // stage consumed (one MMA commit)
    uint64_t* rfull = empty + C::S;
    uint64_t* rempty = rfull + C::RS;
    uint64_t* tfull = rempty + C::RS;
    uint64_t* xs_ready = tfull + 1;                                     // s_xscale filled
    uint32_t* tslot = reinterpret_cast<uint32_t*>(xs_ready + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    static_assert(!(MOE && SPLIT), "the grouped form does not split K");
    // tile (row tile bx, token tile by) and K slice z of ks; the split form
    // walks a 1-D grid: n_full whole tiles, then the rest in ks slices each
    int bx = (int)blockIdx.x, by = (int)blockIdx.y, z = 0, ks = 1;
    int64_t split_tile = 0;   // the tile's index among the split ones
    if constexpr (SPLIT) {
        const int64_t b = blockIdx.x;
        int64_t t;
        if (b < fp.n_full) {
            t = b;
        } else {
            ks = fp.ks;
            split_tile = (b - fp.n_full) / ks;
            z = (int)((b - fp.n_full) % ks);
            t = fp.n_full + split_tile;
        }
        bx = (int)(t % fp.ntile_n);
        by = (int)(t / fp.ntile_n);
    }
    const int64_t n0 = (int64_t)bx * 128;   // first output feature of the tile
    // this CTA's super-blocks [kb0, kb0 + nkb) of the K slice z
    const int kb0 = (int)((int64_t)z * fp.KB / ks);
    const int nkb = (int)((int64_t)(z + 1) * fp.KB / ks) - kb0, nk = 4 * nkb;
    // tile geometry: weight row coordinate, activation row coordinate, valid token columns
    int64_t wrow0, brow0, t0 = 0;
    int cols, expert = 0, gstart = 0;
    if constexpr (MOE) {
        pdl_wait();   // the work items and gathered rows come from the kernels before
        if ((int)blockIdx.y >= *fp.ntiles) return;   // uniform exit before any shared state exists
        const int4 tl = fp.tiles[blockIdx.y];
        expert = tl.x;
        gstart = fp.offsets[tl.x] + tl.y;
        wrow0 = (int64_t)tl.x * fp.N + n0;
        brow0 = gstart;
        cols = tl.z;
    } else {
        t0 = (int64_t)by * BN;
        wrow0 = n0;
        brow0 = t0;
        cols = (int)min((int64_t)BN, fp.M - t0);
    }
    // MMA width: the tile's valid token columns rounded up to 16, so an
    // underfilled tile issues only the MMA columns it needs
    const int n_mma = fp.full_width ? BN : min(BN, (cols + 15) & ~15);
    // the power-of-two scales of the tile's activation rows, staged for the
    // epilogue by the activation producer's warp (off the start-up path)
    __shared__ float s_xscale[BN];

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::S; ++s) { mbar_init(&full[s], DW + 1); mbar_init(&empty[s], NI); }
        for (int s = 0; s < C::RS; ++s) { mbar_init(&rfull[s], 1); mbar_init(&rempty[s], DW); }
        mbar_init(tfull, NI);
        mbar_init(xs_ready, 32);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tslot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0) {
        // raw super-blocks, as far ahead as the raw ring allows
        if (lane == 0) {
            prefetch_tmap(&tmW0);
            for (int kl = 0; kl < nkb; ++kl) {
                const int kb = kb0 + kl, rs = kl % C::RS;
                if (!mbar_wait(&rempty[rs], ((kl / C::RS) & 1) ^ 1, fp.status)) break;
                uint8_t* dst = sR + rs * RAW;
                mbar_arrive_expect_tx(&rfull[rs], RAW);
                if constexpr (PLANES) {
                    tma_load_2d(dst, &tmW0, kb * 64, (int)wrow0, &rfull[rs]);                     // QL: 128 B per row
                    tma_load_2d(dst + 128 * 128, &tmW1, kb * 32, (int)wrow0, &rfull[rs]);         // QH: 64 B
                    tma_load_2d(dst + 128 * 192, &tmW2, kb * 8, (int)wrow0, &rfull[rs]);          // SC: 16 B
                    tma_load_2d(dst + 128 * 208, &tmW3, ((2 * kb) & ~15) / 2, (int)wrow0, &rfull[rs]);  // D: 16 B
                } else if constexpr (QT == GGUF_Q6_K || k23(QT)) {
                    constexpr int BB = block_bytes(QT);
                    tma_load_2d(dst, &tmW0, ((BB * kb) & ~15) / 2, (int)wrow0, &rfull[rs]);
                } else {   // columns of a multiple of 16 bytes: boxed from their own start
                    tma_load_2d(dst, &tmW0, kb * (col_bytes(QT) / 2), (int)wrow0, &rfull[rs]);
                }
            }
        }
    } else if (warp == 2) {
        // the activation tile of every 64-value k step, as far ahead as the ring
        // allows; first the tile's row scales into shared memory (all lanes)
        if (lane == 0) prefetch_tmap(&tmB);
        pdl_wait();   // the f16 activations and their scales come from the kernel before this one
        for (int i = lane; i < BN; i += 32)
            s_xscale[i] = i < cols ? fp.xscale[MOE ? (int64_t)gstart + i : t0 + i] : 1.f;
        mbar_arrive(xs_ready);
        if (lane == 0) {
            for (int i = 0; i < nk; ++i) {
                const int s = i % C::S;
                if (!mbar_wait(&empty[s], ((i / C::S) & 1) ^ 1, fp.status)) break;
                mbar_arrive_expect_tx(&full[s], C::B_BYTES);
                tma_load_2d(sB + s * C::B_BYTES, &tmB, (4 * kb0 + i) * 64, (int)brow0, &full[s]);
            }
        }
    } else if (warp == 1 || warp >= 3 + DW) {
        // issuer j: the 16-value k slices [j*4/NI, (j+1)*4/NI) of every step,
        // into accumulator j
        if (lane == 0) {
            constexpr int KS = 4 / NI;
            const int j = warp == 1 ? 0 : warp - (2 + DW);
            const uint32_t d = tmem + (uint32_t)(j * BN);
            const uint32_t idesc = idesc_f16(128, n_mma, 0);
            // B descriptor of stage s, k slice k: the start-address field is
            // linear in the address (+B_BYTES/16 per stage, +2 per 16 values)
            const uint64_t bdesc0 = sw128_desc(smem_u32(sB));
            for (int i = 0; i < nk; ++i) {
                const int s = i % C::S;
                if (!mbar_wait(&full[s], (i / C::S) & 1, fp.status)) break;
                tc_fence_after();
                const uint32_t a0 = tmem + (uint32_t)(C::A_COL0 + s * C::A_COLS);
                const uint64_t b0 = bdesc0 + (uint64_t)(s * (C::B_BYTES >> 4));
#pragma unroll
                for (int k = j * KS; k < (j + 1) * KS; ++k)
                    umma_f16_ts(d, a0 + 8 * k, b0 + 2 * k, idesc, (i | (k - j * KS)) != 0);
                umma_commit(&empty[s]);
            }
            umma_commit(tfull);
        }
    } else {
        // decoders: warp w handles the 32 rows of TMEM lane quarter w % 4 (row
        // r = 32 * (w % 4) + lane) and part (w - 3) / 4 of every k step: a half
        // hf (8 warps) or a quarter (hf, hh) (16 warps) of its 64 values
        const int part = (warp - 3) >> 2, r = 32 * (warp & 3) + lane;
        const int hf = DW == 16 ? part >> 1 : part, hh = DW == 16 ? part & 1 : 0;
        const uint32_t t_lane = (uint32_t)(32 * (warp & 3)) << 16;
        int i = 0;
        bool ok = true;
        for (int kl = 0; kl < nkb && ok; ++kl) {
            const int kb = kb0 + kl, rs = kl % C::RS;
            ok = mbar_wait(&rfull[rs], (kl / C::RS) & 1, fp.status);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            const uint32_t slot = smem_u32(sR + rs * RAW);
            uint32_t row = slot + (uint32_t)(r * PITCH);
            if constexpr ((QT == GGUF_Q6_K && !PLANES) || k23(QT)) row += (uint32_t)((block_bytes(QT) * kb) & 15);
            constexpr bool STATE = QT == GGUF_Q4_K || QT == GGUF_Q5_K || PLANES;
            KbState<QT, LAYOUT> st;
            if constexpr (STATE) st.prepare(row, slot, r, hf, kb, DW == 16 ? hh : -1);
            // DB consecutive k steps per round: their stages are claimed
            // together and decoded side by side, so one warp's chain of
            // waits, loads and the TMEM store completion is paid once per DB
            // steps (the step rate is bound by that chain, not by issue slots)
#pragma unroll
            for (int q = 0; q < 4; q += DB, i += DB) {
                bool got = true;
#pragma unroll
                for (int d = 0; d < DB; ++d)
                    got = got && mbar_wait(&empty[(i + d) % C::S], (((i + d) / C::S) & 1) ^ 1, fp.status);
                ok = got;
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();   // the MMAs that read these stages have completed
                if constexpr (DW == 16) {
                    uint32_t v[DB][8];
#pragma unroll
                    for (int d = 0; d < DB; ++d) {
                        uint4 out[2];
                        decode_quarter<QT, LAYOUT>(st, row, slot, r, q + d, hf, hh, out);
                        v[d][0] = out[0].x; v[d][1] = out[0].y; v[d][2] = out[0].z; v[d][3] = out[0].w;
                        v[d][4] = out[1].x; v[d][5] = out[1].y; v[d][6] = out[1].z; v[d][7] = out[1].w;
                    }
#pragma unroll
                    for (int d = 0; d < DB; ++d) {   // values 32hf + 16hh .. +15 of step i + d
                        const uint32_t ta = tmem + t_lane + (uint32_t)(C::A_COL0 + ((i + d) % C::S) * C::A_COLS);
                        tmem_st8(ta + (uint32_t)(16 * hf + 8 * hh), v[d]);
                    }
                } else if constexpr (STATE) {
#pragma unroll
                    for (int d = 0; d < DB; ++d) {   // values 32hf .. +31 of step i + d: two quarters
                        uint4 out[4];
                        decode_quarter<QT, LAYOUT, true>(st, row, slot, r, q + d, hf, 0, out);
                        decode_quarter<QT, LAYOUT, true>(st, row, slot, r, q + d, hf, 1, out + 2);
                        const uint32_t v[16] = {out[0].x, out[0].y, out[0].z, out[0].w, out[1].x, out[1].y,
                                                out[1].z, out[1].w, out[2].x, out[2].y, out[2].z, out[2].w,
                                                out[3].x, out[3].y, out[3].z, out[3].w};
                        const uint32_t ta = tmem + t_lane + (uint32_t)(C::A_COL0 + ((i + d) % C::S) * C::A_COLS);
                        tmem_st16(ta + (uint32_t)(16 * hf), v);
                    }
                } else {
#pragma unroll
                    for (int d = 0; d < DB; ++d) {   // values 32hf .. +31 of step i + d
                        uint4 out[4];
                        decode32<QT, LAYOUT>(row, slot, r, q + d, hf, kb, out);
                        const uint32_t v[16] = {out[0].x, out[0].y, out[0].z, out[0].w, out[1].x, out[1].y,
                                                out[1].z, out[1].w, out[2].x, out[2].y, out[2].z, out[2].w,
                                                out[3].x, out[3].y, out[3].z, out[3].w};
                        const uint32_t ta = tmem + t_lane + (uint32_t)(C::A_COL0 + ((i + d) % C::S) * C::A_COLS);
                        tmem_st16(ta + (uint32_t)(16 * hf), v);
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int d = 0; d < DB; ++d) mbar_arrive(&full[(i + d) % C::S]);
                }
            }
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&rempty[rs]);
        }
        // epilogue: decoder warp w reads TMEM lane quarter (w % 4) and column
        // group (w - 3) / 4 of DW / 4 groups of 16-column chunks
        constexpr int G = DW / 4, CH = BN / 16;
        const int qd = warp & 3, grp = (warp - 3) >> 2;
        const int64_t n = n0 + 32 * qd + lane;
        const bool ep_ok = __all_sync(0xffffffffu, mbar_wait(tfull, 0, fp.status) && mbar_wait(xs_ready, 0, fp.status));
        pdl_wait();   // the split tickets are zeroed by the kernel before this one
        // split K: this slice's sums go to its slot [BN][128] of the tile
        float* const slots = SPLIT ? fp.partial + split_tile * ks * (BN * 128) : nullptr;
        if (ep_ok) {
            tc_fence_after();
#pragma unroll 1
            for (int c = grp * CH / G; c < (grp + 1) * CH / G; ++c) {
                if (16 * c >= n_mma) break;   // columns past the MMA width hold nothing
                uint32_t v[16];
                tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) + 16 * c, v);
                tmem_ld_wait();
                tmem_ld_regs(v);
#pragma unroll
                for (int j = 1; j < NI; ++j) {   // the other issuers' partial sums, one at a time
                    uint32_t u[16];
                    tmem_ld16(tmem + ((uint32_t)(32 * qd) << 16) + j * BN + 16 * c, u);
                    tmem_ld_wait();
                    tmem_ld_regs(u);
#pragma unroll
                    for (int e = 0; e < 16; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) + __uint_as_float(u[e]));
                }
                if (SPLIT && ks > 1) {
                    // column-major slot: a warp's 32 rows of a column are one 128-byte line
                    float* dst = slots + (int64_t)z * (BN * 128) + (16 * c) * 128 + 32 * qd + lane;
#pragma unroll
                    for (int j = 0; j < 16; ++j) dst[j * 128] = __uint_as_float(v[j]);
                } else if (n < fp.N) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int col = 16 * c + j;
                        if (col < cols) {
                            // output row: token m (dense) or the routed entry (grouped)
                            const int64_t orow = MOE ? (int64_t)fp.rows[gstart + col] : t0 + col;
                            float o = __uint_as_float(v[j]) * s_xscale[col];
                            if (fp.residual) o += load_act(fp.residual, fp.ydt, orow * fp.N + n);
                            store_out(fp.y, fp.ydt, orow * fp.N + n, o);
                        }
                    }
                }
            }
        }
        if (SPLIT && ks > 1) {   // uniform across the CTA
            // the last slice to finish the tile adds the slots in slice order
            // (a fixed order: the result does not depend on which CTA is last)
            volatile int* ticket = reinterpret_cast<volatile int*>(tslot + 1);
            __threadfence();
            named_bar_sync(1, DW * 32);
            if (warp == 3 && lane == 0) *ticket = ep_ok ? atomicAdd(&fp.tickets[split_tile], 1) : -1;
            named_bar_sync(1, DW * 32);
            if (*ticket == ks - 1) {
                __threadfence();
#pragma unroll 1
                for (int c = grp * CH / G; c < (grp + 1) * CH / G; ++c) {
                    if (16 * c >= n_mma || n >= fp.N) break;
                    // a slot's 16 columns are loaded together: one L2 round trip per slot
                    float acc[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) acc[j] = 0.f;
                    const float* src = slots + (16 * c) * 128 + 32 * qd + lane;
#pragma unroll 1
                    for (int q = 0; q < ks; ++q) {
                        float t[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) t[j] = __ldcg(src + (int64_t)q * (BN * 128) + j * 128);
#pragma unroll
                        for (int j = 0; j < 16; ++j) acc[j] += t[j];
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int col = 16 * c + j;
                        if (col < cols) {
                            const int64_t orow = t0 + col;
                            float o = acc[j] * s_xscale[col];
                            if (fp.residual) o += load_act(fp.residual, fp.ydt, orow * fp.N + n);
                            store_out(fp.y, fp.ydt, orow * fp.N + n, o);
                        }
                    }
                }
            }
        }
        (void)expert;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

// Tile plan: token-tile width BN and K split ks with the least estimated
// time, in k steps per round of CTAs times the per-step cost.  A step's cost
// is nearly flat in BN (the step rate is set by the decoder warps, not by the
// MMA width): ~ (bn + 1150).  Every CTA also pays ~24 steps of fixed cost
// (start-up until the first blocks are decoded, epilogue, the gap before the
// next round), and a K split ~8 more (partial tile out, the last slice reads
// the slots back).  Measured on GB300: splitting pays where the tiles alone
// leave most SMs idle (N = 2048: 16 row tiles, 49 -> 28 us at M = 128) and
// loses at N = 14336 (M = 512: 67 us unsplit, 79 us in halves).  A candidate
// must beat the best so far by 3 %, so ties keep the smaller tile and split.
// Two kinds of split: every tile in ks slices (n_full = 0), or only the tiles
// of the last, partial round (the first n_full whole, the rest in ks slices,
// which fill the SMs the partial round would leave idle: 224 tiles at M = 512
// are one round of 152 whole tiles and 72 tiles in halves).
struct FusedPlan {
    int bn, ks;
    int64_t n_full;   // tiles kept whole (in launch order) when ks > 1
};
FusedPlan plan_fused(int64_t N, int64_t M, int64_t KB, int num_sms) {
    FusedPlan best{32, 1, 0};
    double best_cost = 1e300;
    const int64_t steps = 4 * KB;
    auto consider = [&](double cost, FusedPlan p) {
        if (cost < best_cost * 0.97) { best_cost = cost; best = p; }
    };
    for (int bn : {32, 64, 128, 256}) {
        const double step_cost = (double)(std::min<int64_t>(bn, M) + 1150);
        const int64_t tiles = ceil_div(N, 128) * ceil_div(M, bn);
        for (int ks = 1; ks <= 16; ++ks) {
            if (ks > KB || (ks > 1 && steps / ks < 8)) break;
            const double per = (double)(ceil_div(steps, ks) + 24 + (ks > 1 ? 8 : 0)) * step_cost;
            consider((double)ceil_div(tiles * ks, num_sms) * per, {bn, ks, 0});
        }
        // whole rounds, then the partial round's tiles split to fill the SMs
        const int64_t rounds = tiles / num_sms, tail = tiles - rounds * num_sms;
        if (rounds >= 1 && tail > 0) {
            for (int ks = 2; ks <= 16 && ks <= KB && steps / ks >= 8 && tail * ks <= num_sms; ++ks) {
                const double cost = ((double)rounds * (steps + 24) + (double)(ceil_div(steps, ks) + 24 + 8)) * step_cost;
                consider(cost, {bn, ks, rounds * num_sms});
            }
        }
    }
    return best;
}

// Whether format QT (layout LAYOUT) can run two CTAs per SM at BN = 128: half
// of shared memory still holds four activation stages and two raw slots.
// Used by the grouped (MoE) form only: dense tiles measured slower two per SM
// (Q5_K 14336 x 4096, M = 8 / 128 / 512: 26.4 -> 31.7, 28.2 -> 38.8, 63.7 ->
// 87.4 us) -- half of shared memory leaves two or three raw slots, too few to
// cover the weight stream's latency over a 64-step tile, while MoE work items
// (K = 2048, a few token columns) gain more from overlapping one CTA's
// start-up and epilogue with the other's decoding.
template <int QT, int LAYOUT>
constexpr bool two_ctas_fit() {
    using C2 = FusedCfg<128, raw_slot_bytes(QT, LAYOUT), 2>;
    return C2::OK && C2::S >= 4;
}

// Workspace layout of the fused GEMM: F16 activations | split-K slots | tickets.
struct FusedWorkspace {
    size_t act, scale, partial, tickets, total;   // act: bytes of the f16 copy; the others are offsets
};
FusedWorkspace fused_workspace(int64_t N, int64_t K, int64_t M, const FusedPlan& pl) {
    FusedWorkspace w{};
    w.act = (size_t)act_copy_bytes(M, K);
    w.scale = w.act;
    w.total = w.act + (size_t)act_scale_bytes(M);
    if (pl.ks > 1) {
        const int64_t split = ceil_div(N, 128) * ceil_div(M, pl.bn) - pl.n_full;   // tiles in slices
        w.partial = w.total;
        w.total += (size_t)(ceil_div(split * pl.ks * pl.bn * 128 * 4, 256) * 256);
        w.tickets = w.total;
        w.total += (size_t)(ceil_div(split * 4, 256) * 256);
    }
    return w;
}

template <int QT, int LAYOUT, int BN, bool MOE = false, bool SPLIT = false, int CTAS = 1>
cudaError_t launch_fused(const CUtensorMap* w, const CUtensorMap& b, const FusedParams& fp, cudaStream_t s,
                         int grid_y = 0) {
    using C = FusedCfg<BN, raw_slot_bytes(QT, LAYOUT), CTAS>;
    const int smem = C::SMEM;
    auto k = fused_tc_kernel<QT, LAYOUT, BN, MOE, SPLIT, CTAS>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (CTAS > 1 &&   // the whole carveout to shared memory, so that two CTAs fit
        (e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
        return e;
    dim3 grid((unsigned)ceil_div(fp.N, 128), MOE ? (unsigned)grid_y : (unsigned)ceil_div(fp.M, BN));
    if (SPLIT) {
        const int64_t tiles = ceil_div(fp.N, 128) * ceil_div(fp.M, BN);
        grid = dim3((unsigned)(fp.n_full + (tiles - fp.n_full) * fp.ks));
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(fused_threads(QT, LAYOUT, BN, CTAS));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = fp.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, w[0], w[1], w[2], w[3], b, fp);
}

template <int QT, int LAYOUT>
cudaError_t launch_bn(int bn, const CUtensorMap* w, const CUtensorMap& b, const FusedParams& fp, cudaStream_t s) {
    const bool split = fp.ks > 1;
    switch (bn) {
        case 256: return split ? launch_fused<QT, LAYOUT, 256, false, true>(w, b, fp, s)
                               : launch_fused<QT, LAYOUT, 256>(w, b, fp, s);
        case 128: return split ? launch_fused<QT, LAYOUT, 128, false, true>(w, b, fp, s)
                               : launch_fused<QT, LAYOUT, 128>(w, b, fp, s);
        case 64: return split ? launch_fused<QT, LAYOUT, 64, false, true>(w, b, fp, s)
                              : launch_fused<QT, LAYOUT, 64>(w, b, fp, s);
        default: return split ? launch_fused<QT, LAYOUT, 32, false, true>(w, b, fp, s)
                              : launch_fused<QT, LAYOUT, 32>(w, b, fp, s);
    }
}

// The grouped (MoE) form: two CTAs per SM where half of shared memory still
// holds four activation stages and two raw slots (GGUF_MM_MOE_CTAS=1 in the
// environment, read at each call, keeps one: a comparison arm).
template <int QT>
cudaError_t launch_grouped(const CUtensorMap* w, const CUtensorMap& b, const FusedParams& fp, cudaStream_t s,
                           int grid_y) {
    if constexpr (two_ctas_fit<QT, 0>()) {
        const char* env = std::getenv("GGUF_MM_MOE_CTAS");
        if (!(env && env[0] == '1')) return launch_fused<QT, 0, 128, true, false, 2>(w, b, fp, s, grid_y);
    }
    return launch_fused<QT, 0, 128, true>(w, b, fp, s, grid_y);
}

}  // namespace

size_t gemm_workspace_bytes(int, int64_t N, int64_t K, int64_t M, int num_sms) {
    if (K % 256 != 0) return (size_t)(ceil_div(M * K * 2, 256) * 256);
    return fused_workspace(N, K, M, plan_fused(N, M, K / 256, num_sms)).total;
}

int gemm_fused_run(const void* w, int qtype, int layout, int64_t N, int64_t K, const void* x, int xdt, int64_t M,
                   const void* residual, void* y, int ydt, void* workspace, int num_sms, int* status,
                   cudaStream_t stream, int pdl) {
    if (K % 256 != 0) return GGUF_ERR_UNSUPPORTED;
    const int64_t KB = K / 256;
    // 16-byte row strides for TMA: raw Q6_K and Q3_K rows need K % 2048, Q2_K K % 1024
    if ((qtype == GGUF_Q6_K || qtype == GGUF_Q3_K) && KB % 8 != 0) return GGUF_ERR_UNSUPPORTED;
    if (qtype == GGUF_Q2_K && KB % 4 != 0) return GGUF_ERR_UNSUPPORTED;
    if (N > INT32_MAX || M > INT32_MAX || KB > (1 << 20)) return GGUF_ERR_UNSUPPORTED;
    const FusedPlan pl = plan_fused(N, M, KB, num_sms);
    const FusedWorkspace wl = fused_workspace(N, K, M, pl);
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    int* tickets = pl.ks > 1 ? reinterpret_cast<int*>(wsb + wl.tickets) : nullptr;
    const int ntiles = (int)(ceil_div(N, 128) * ceil_div(M, pl.bn) - pl.n_full);   // tiles in slices
    float* xscale = reinterpret_cast<float*>(wsb + wl.scale);
    if (convert_activations(x, xdt, M, K, workspace, GGUF_DT_F16, xscale, num_sms, stream,
                            reinterpret_cast<uint32_t*>(tickets), tickets ? ntiles : 0) != cudaSuccess)
        return GGUF_ERR_CUDA;

    const int bb = block_bytes(qtype) * (block32(qtype) ? 8 : 1);   // bytes of one 256-value column
    const int64_t rb = KB * bb;
    CUtensorMap tw[4];
    std::memset(tw, 0, sizeof(tw));
    int st;
    const CUtensorMapDataType u16 = CU_TENSOR_MAP_DATA_TYPE_UINT16;
    const CUtensorMapSwizzle none = CU_TENSOR_MAP_SWIZZLE_NONE;
    if (qtype == GGUF_Q6_K && layout == GGUF_LAYOUT_Q6K_PLANES) {
        const int64_t nblk = N * KB;
        const uint8_t* p = static_cast<const uint8_t*>(w);
        // QL (128 B per row) and QH (64 B) land swizzled, so that the decoders'
        // 16-byte reads of 32 consecutive rows spread over all banks
        if ((st = make_tmap_2d(&tw[0], p, u16, 2, 64 * KB, N, 128 * KB, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) !=
            GGUF_OK)
            return st;
        if ((st = make_tmap_2d(&tw[1], p + 128 * nblk, u16, 2, 32 * KB, N, 64 * KB, 32, 128,
                               CU_TENSOR_MAP_SWIZZLE_64B)) != GGUF_OK)
            return st;
        if ((st = make_tmap_2d(&tw[2], p + 192 * nblk, u16, 2, 8 * KB, N, 16 * KB, 8, 128, none)) != GGUF_OK) return st;
        if ((st = make_tmap_2d(&tw[3], p + 208 * nblk, u16, 2, KB, N, 2 * KB, 8, 128, none)) != GGUF_OK) return st;
    } else {
        const uint32_t box = (uint32_t)raw_pitch(qtype, 0) / 2;
        if ((st = make_tmap_2d(&tw[0], w, u16, 2, (uint64_t)rb / 2, N, rb, box, 128, none)) != GGUF_OK) return st;
        tw[1] = tw[2] = tw[3] = tw[0];
    }
    const int bn = pl.bn;
    CUtensorMap tb;
    if ((st = make_tmap_2d(&tb, workspace, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)K, (uint64_t)M,
                           (uint64_t)K * 2, 64, (uint32_t)bn, CU_TENSOR_MAP_SWIZZLE_128B)) != GGUF_OK)
        return st;
    FusedParams fp{N, M, (int)KB, residual, y, ydt, status, nullptr, nullptr, nullptr, nullptr, 0,
                   pl.ks, pl.ks > 1 ? reinterpret_cast<float*>(wsb + wl.partial) : nullptr, tickets,
                   (int)pl.n_full, (int)ceil_div(N, 128), xscale,
                   // as a dependent launch where whole tiles remain (measured on GB300: Q5_K /
                   // Q6_K planes 14336 x 4096 M = 512 67.2 -> 64.2 / 64.7 -> 61.9 us, Q8_0
                   // 2048 x 8192 M = 4096 138.3 -> 134.1 us), not when every tile is split
                   // along K (M = 128 / 512 there: 25.7 -> 28.6 / 37.8 -> 40.3 us)
                   (pdl && !(pl.ks > 1 && pl.n_full == 0)) ? 1 : 0};
    cudaError_t e = cudaErrorInvalidValue;
    switch (qtype) {
        case GGUF_Q4_0: e = launch_bn<GGUF_Q4_0, 0>(bn, tw, tb, fp, stream); break;
        case GGUF_Q4_1: e = launch_bn<GGUF_Q4_1, 0>(bn, tw, tb, fp, stream); break;
        case GGUF_Q5_0: e = launch_bn<GGUF_Q5_0, 0>(bn, tw, tb, fp, stream); break;
        case GGUF_Q5_1: e = launch_bn<GGUF_Q5_1, 0>(bn, tw, tb, fp, stream); break;
        case GGUF_Q8_0: e = launch_bn<GGUF_Q8_0, 0>(bn, tw, tb, fp, stream); break;
        case GGUF_Q2_K: e = launch_bn<GGUF_Q2_K, 0>(bn, tw, tb, fp, stream); break;
        case GGUF_Q3_K: e = launch_bn<GGUF_Q3_K, 0>(bn, tw, tb, fp, stream); break;
        case GGUF_Q4_K: e = launch_bn<GGUF_Q4_K, 0>(bn, tw, tb, fp, stream); break;
        case GGUF_Q5_K: e = launch_bn<GGUF_Q5_K, 0>(bn, tw, tb, fp, stream); break;
        case GGUF_Q6_K:
            e = layout == GGUF_LAYOUT_Q6K_PLANES ? launch_bn<GGUF_Q6_K, 1>(bn, tw, tb, fp, stream)
                                                 : launch_bn<GGUF_Q6_K, 0>(bn, tw, tb, fp, stream);
            break;
    }
    return e == cudaSuccess ? GGUF_OK : GGUF_ERR_CUDA;
}

int grouped_gemm_run(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K, const void* xg,
                     const float* xscale, int64_t rows_cap, const int4* tiles, const int* ntiles, const int* offsets,
                     const int* rows, int64_t max_tiles, const void* residual, void* y, int ydt, int* status,
                     cudaStream_t stream, int pdl) {
    const int64_t KB = K / 256;
    // 16-byte row strides for TMA: raw Q6_K and Q3_K rows need K % 2048, Q2_K K % 1024
    if ((qtype == GGUF_Q6_K || qtype == GGUF_Q3_K) && KB % 8 != 0) return GGUF_ERR_UNSUPPORTED;
    if (qtype == GGUF_Q2_K && KB % 4 != 0) return GGUF_ERR_UNSUPPORTED;
    if (max_tiles > 65535 || KB > (1 << 20)) return GGUF_ERR_UNSUPPORTED;
    const int bb = block_bytes(qtype) * (block32(qtype) ? 8 : 1);
    const int64_t rb = KB * bb;
    CUtensorMap tw[4];
    std::memset(tw, 0, sizeof(tw));
    // every expert's [N, rb] block rows back to back: one [E*N, rb] tensor
    const uint32_t box = (uint32_t)raw_pitch(qtype, 0) / 2;
    int st = make_tmap_2d(&tw[0], w_experts, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, (uint64_t)rb / 2,
                          (uint64_t)(n_expert * N), rb, box, 128, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != GGUF_OK) return st;
    tw[1] = tw[2] = tw[3] = tw[0];
    CUtensorMap tb;
    if ((st = make_tmap_2d(&tb, xg, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (uint64_t)K, (uint64_t)rows_cap,
                           (uint64_t)K * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B)) != GGUF_OK)
        return st;
    // GGUF_MM_MOE_FULL_TILES=1: every tile's MMA at the full 128 columns, as
    // without the tile-skip (a comparison arm for measurement; same output)
    const char* full = std::getenv("GGUF_MM_MOE_FULL_TILES");
    FusedParams fp{N, rows_cap, (int)KB, residual, y, ydt, status, tiles, ntiles, offsets, rows,
                   (full && full[0] == '1') ? 1 : 0, 1, nullptr, nullptr, 0, 0, xscale, pdl};
    const int gy = (int)max_tiles;
    cudaError_t e = cudaErrorInvalidValue;
    switch (qtype) {
        case GGUF_Q4_0: e = launch_grouped<GGUF_Q4_0>(tw, tb, fp, stream, gy); break;
        case GGUF_Q4_1: e = launch_grouped<GGUF_Q4_1>(tw, tb, fp, stream, gy); break;
        case GGUF_Q5_0: e = launch_grouped<GGUF_Q5_0>(tw, tb, fp, stream, gy); break;
        case GGUF_Q5_1: e = launch_grouped<GGUF_Q5_1>(tw, tb, fp, stream, gy); break;
        case GGUF_Q8_0: e = launch_grouped<GGUF_Q8_0>(tw, tb, fp, stream, gy); break;
        case GGUF_Q2_K: e = launch_grouped<GGUF_Q2_K>(tw, tb, fp, stream, gy); break;
        case GGUF_Q3_K: e = launch_grouped<GGUF_Q3_K>(tw, tb, fp, stream, gy); break;
        case GGUF_Q4_K: e = launch_grouped<GGUF_Q4_K>(tw, tb, fp, stream, gy); break;
        case GGUF_Q5_K: e = launch_grouped<GGUF_Q5_K>(tw, tb, fp, stream, gy); break;
        case GGUF_Q6_K: e = launch_grouped<GGUF_Q6_K>(tw, tb, fp, stream, gy); break;
    }
    return e == cudaSuccess ? GGUF_OK : GGUF_ERR_CUDA;
}

}  // namespace gg
