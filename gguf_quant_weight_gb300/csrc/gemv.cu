// Decode GEMV on GGUF blocks: Y[m, n] = sum_k X[m, k] W[n, k] (+ residual).
//
// OpenVINO PR #39119 "FullyConnectedGGUF", "Implementation", GEMV row: the
// activations are quantized per 32 values to int8 (Q8-style, one f32 scale per
// block) and every weight sub-block is dotted in integers straight against its
// GGUF bytes; the float scales are applied once per sub-block.
//
// GB300 shape of it (two 256-thread CTAs per SM, rows of W dealt to warps):
//  * at entry every warp requests the bytes of all its weight rows (up to a
//    ring of R row slots in shared memory) with 16-byte coalesced async copies,
//    so the whole matrix is in flight from the first microsecond; then the CTA
//    tells the next kernel on the stream it may launch (programmatic dependent
//    launch), so the next call's weight stream starts while this one finishes;
//  * prologue, after waiting for the producer of X: the CTA quantizes the M
//    activation rows into shared memory (codes, per-32 scale d_a, code sums);
//  * a lane owns one "unit" of a row: half a 256-value super-block (or one
//    Q8_0 block); a warp covers a whole row (or several rows when K is small);
//    a lane's K slice never changes from row to row, so its activation codes
//    and scales are loaded into registers once (M = 1, 2) or read from
//    bank-conflict-free shared memory (larger M);
//  * dp4a on 4 weights x 4 codes, integer sub-block scaling, one int->float per
//    activation block, a (segmented) warp-shuffle reduction, and the residual
//    Add fused into the store.
#include "common.cuh"
#include "formats.cuh"
#include "gemv.cuh"
#include <cstdlib>
#include <type_traits>

namespace gg {

namespace {

constexpr int kThreads = 256;

// Activation codes of row m live at qa + m*qa_row_stride(K), element k at byte
// k + 16*(k/128): a lane reads the 16-byte pieces of one 128-value unit, and
// the 16-byte pad after every 128 codes puts the 8 lanes of each quarter-warp
// phase on different 4-bank groups (conflict-free 16-byte loads).
__host__ __device__ constexpr int64_t qa_row_stride(int64_t K) { return K + 16 * ceil_div(K, 128); }
__device__ __forceinline__ uint32_t qa_pos(uint32_t k) { return k + ((k >> 7) << 4); }

// Per 32-value activation block and row: {d_a (f32), d_a * s (f32), s_lo, s_hi}
// with s = sum of the 32 codes and s_lo / s_hi the sums of its two halves.
struct Shared {
    uint32_t qa;     // shared address of the codes
    uint32_t ds;     // shared address of the per-block entries (16 bytes each)
    uint32_t stage;  // shared address of the per-warp staging buffers
    uint32_t qa_row; // bytes per code row
};

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts64(uint32_t a, uint32_t x, uint32_t y) {
    asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(a), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ float i2f(int v) { return (float)v; }


__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Nearest integer, halves away from zero, for |y| <= 127.5: y + copysign(0.5, y)
// rounded toward zero, then truncated.  Rounding the sum toward zero never
// carries it across an integer (integers are representable), so the result is
// floor(|y| + 0.5) with y's sign.
__device__ __forceinline__ int round_half_away(float y) {
    return __float2int_rz(__fadd_rz(y, copysignf(0.5f, y)));
}

__device__ __forceinline__ uint32_t comp(const uint4& v, int i) {
    return (i & 3) == 0 ? v.x : (i & 3) == 1 ? v.y : (i & 3) == 2 ? v.z : v.w;
}

// ------------------------------------------------------------------ activation quantizer
// Per 32 values: amax, d_a = amax/127 (IEEE f32 divide), id = 1/d_a (0 for an
// all-zero block), q = round-half-away(clamp(x*id, -127, 127)), s = sum q.
// The image it writes is the GEMV's shared-memory layout byte for byte:
// [M][qa_row_stride(K)] codes, then [M][K/32] entries of 16 bytes
// {d_a, d_a*s, s_lo, s_hi}.
//
// Four threads per 32-value block (8 values each, lanes 4j..4j+3 of a warp);
// the block's amax and code sums are combined with shuffles inside the group,
// so every lane of the warp must take part (on = false for padding lanes).

// The 8 activation values at element offset `off` of X, as f32.
__device__ __forceinline__ void load_quarter(const GemvParams& p, bool on, int64_t off, float (&v)[8]) {
    if (!on) {   // padding lane: any finite non-zero block (nothing is stored)
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = 1.f;
    } else if (p.xdt == GGUF_DT_F32) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.x) + off);
        const float4 a = src[0], c = src[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
    } else {
        const uint4 t = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) + off);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t wv = comp(t, j);
            if (p.xdt == GGUF_DT_BF16) {
                v[2 * j] = __uint_as_float(wv << 16);
                v[2 * j + 1] = __uint_as_float(wv & 0xFFFF0000u);
            } else {
                v[2 * j] = f16_bits_to_float(wv & 0xFFFFu);
                v[2 * j + 1] = f16_bits_to_float(wv >> 16);
            }
        }
    }
}

// Quantizes one quarter: its 8 codes in word[0..1] and the block's entry
// {d_a, d_a * s, s of quarters 0-1, s of quarters 2-3} (complete in the
// lanes of quarter 0 and 2; quarter 0's is the one stored).
__device__ __forceinline__ void quant_core(const float (&v)[8], uint32_t (&word)[2], uint4& entry) {
    // amax propagates NaN (a NaN anywhere in the block makes d_a NaN)
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = max_nan(amax, fabsf(v[i]));
    amax = max_nan(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max_nan(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = amax / 127.0f;
    const float id = d != 0.f ? 1.0f / d : 0.f;
    // clamp, then round (NaN clamps to -127); no branch, so the quarters of a
    // round interleave
    int q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = round_half_away(fminf(fmaxf(v[i] * id, -127.f), 127.f));
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        // cvt.pack.sat.s8.s32.b32 d, a, b, c: d = (c << 16) | (a << 8) | b
        // (a, b saturated to s8), so the inner pair becomes the upper bytes
        uint32_t hi;
        asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, 0;" : "=r"(hi) : "r"(q[4 * j + 3]), "r"(q[4 * j + 2]));
        asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(word[j]) : "r"(q[4 * j + 1]), "r"(q[4 * j]), "r"(hi));
    }
    const int s8 = dp4a(word[0], 0x01010101u, dp4a(word[1], 0x01010101u, 0));
    const int s_pair = s8 + __shfl_xor_sync(0xffffffffu, s8, 1);   // s_lo (quarters 0,1) or s_hi (2,3)
    const int s_other = __shfl_xor_sync(0xffffffffu, s_pair, 2);
    const int s = s_pair + s_other;
    entry = make_uint4(__float_as_uint(d), __float_as_uint(d * (float)s), (uint32_t)s_pair, (uint32_t)s_other);
}

// Quantizes one quarter; writes its 8 codes at `codes` and (quarter 0) the
// block's entry at `entry` (generic pointers: global workspace or shared).
__device__ __forceinline__ void quant_values(const float (&v)[8], bool on, int qtr, uint8_t* codes, uint8_t* entry) {
    uint32_t word[2];
    uint4 e;
    quant_core(v, word, e);
    if (on) {
        *reinterpret_cast<uint2*>(codes) = make_uint2(word[0], word[1]);
        if (qtr == 0) *reinterpret_cast<uint4*>(entry) = e;
    }
}

// Quarter qtr of block b of row m, into an image over all of K at img.
__device__ __forceinline__ void quant_quarter(const GemvParams& p, bool on, int m, int b, int qtr, uint8_t* img) {
    const int64_t qa_row = qa_row_stride(p.K);
    const int nb = (int)(p.K / 32);
    float v[8];
    load_quarter(p, on, (int64_t)m * p.K + (int64_t)b * 32 + 8 * qtr, v);
    quant_values(v, on, qtr, img + (int64_t)m * qa_row + qa_pos(b * 32) + 8 * qtr,
                 img + (int64_t)p.M * qa_row + 16 * ((int64_t)m * nb + b));
}

// Threads [0, nthreads) of a block quantize the K slice [k0, k0 + klen) of all
// M rows into an image of that slice at img (codes [M][qa_row_stride(klen)],
// then [M][klen/32] entries).  Each thread takes UNR quarters per round and
// issues all their loads before quantizing any; a warp stops once its first
// quarter of a round is past the end (the group shuffles stay warp-uniform).
template <int UNR>
__device__ __forceinline__ void quantize_slice(const GemvParams& p, int64_t k0, int klen, uint8_t* img, int t0,
                                               int nthreads) {
    const int nb = klen / 32;
    const int per_row = 4 * nb;
    const int quarters = p.M * per_row;
    const uint32_t qa_row = (uint32_t)qa_row_stride(klen);
    const int qtr = t0 & 3;
    for (int base = 0; base < quarters; base += UNR * nthreads) {
        if (base + (t0 & ~31) >= quarters) break;
        float v[UNR][8];
        int m[UNR], b[UNR];
        bool on[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int idx = base + u * nthreads + t0;
            on[u] = idx < quarters;
            const int i = on[u] ? idx : 0;
            m[u] = i / per_row;
            b[u] = (i - m[u] * per_row) >> 2;
            load_quarter(p, on[u], (int64_t)m[u] * p.K + k0 + 32 * b[u] + 8 * qtr, v[u]);
        }
        // straight-line over the UNR quarters (padding quarters compute on
        // zeros and store nothing), so their dependency chains interleave
#pragma unroll
        for (int u = 0; u < UNR; ++u)
            quant_values(v[u], on[u], qtr, img + m[u] * qa_row + qa_pos(32 * b[u]) + 8 * qtr,
                         img + (uint32_t)p.M * qa_row + 16u * (uint32_t)(m[u] * nb + b[u]));
    }
}

// Threads [0, nthreads) of CTA `rank` of a cluster of CL CTAs quantize blocks
// [rank * nb / CL, (rank + 1) * nb / CL) of all M rows (nb = K / 32) and store
// the codes and entries into the image over all of K at shared address `img`
// of every CTA of the cluster (same layout as quantize_slice over all of K),
// so that the CL CTAs share one quantization of X: plain stores into this
// CTA's image, asynchronous stores into the others', each completing its
// bytes on the mbarrier at shared address `bar` of the receiving CTA
// (cluster_xbytes(CL, M, K) bytes per receiver, which its expect_tx counts).
// The caller has made sure that every CTA of the cluster is running and has
// initialised that barrier.
template <int CL, int UNR>
__device__ __forceinline__ void quantize_cluster(const GemvParams& p, uint32_t img, uint32_t bar, int t0,
                                                 int nthreads) {
    const int nb = (int)(p.K / 32), nbs = nb / CL;
    const uint32_t rank = cluster_rank();
    const int b0 = (int)rank * nbs;
    const int per_row = 4 * nbs;
    const int quarters = p.M * per_row;
    const uint32_t qa_row = (uint32_t)qa_row_stride(p.K);
    uint32_t dst[CL], dbar[CL];
#pragma unroll
    for (int c = 0; c < CL; ++c) {
        dst[c] = cluster_map(img, (uint32_t)c);
        dbar[c] = cluster_map(bar, (uint32_t)c);
    }
    const int qtr = t0 & 3;
    for (int base = 0; base < quarters; base += UNR * nthreads) {
        if (base + (t0 & ~31) >= quarters) break;
        float v[UNR][8];
        int m[UNR], b[UNR];
        bool on[UNR];
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            const int idx = base + u * nthreads + t0;
            on[u] = idx < quarters;
            const int i = on[u] ? idx : 0;
            m[u] = i / per_row;
            b[u] = b0 + ((i - m[u] * per_row) >> 2);
            load_quarter(p, on[u], (int64_t)m[u] * p.K + 32 * b[u] + 8 * qtr, v[u]);
        }
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
            uint32_t w[2];
            uint4 e;
            quant_core(v[u], w, e);
            if (on[u]) {
                const uint32_t co = (uint32_t)m[u] * qa_row + qa_pos(32u * (uint32_t)b[u]) + 8u * (uint32_t)qtr;
                const uint32_t eo = (uint32_t)p.M * qa_row + 16u * (uint32_t)(m[u] * nb + b[u]);
                sts64(img + co, w[0], w[1]);
                if (qtr == 0) sts128(img + eo, e);
#pragma unroll
                for (int c = 0; c < CL; ++c) {
                    if ((uint32_t)c == rank) continue;
                    st_async_v2(dst[c] + co, w[0], w[1], dbar[c]);
                    if (qtr == 0) st_async_v4(dst[c] + eo, e, dbar[c]);
                }
            }
        }
    }
}

// Bytes of the activation image a CTA of a cluster of CL receives from the
// other CTAs (their blocks: 32 code bytes and a 16-byte entry each).
__host__ __device__ constexpr int64_t cluster_xbytes(int CL, int64_t M, int64_t K) {
    return (CL - 1) * M * (K / 32 / CL) * 48;
}

// The stand-alone quantizer for the kernels that take the image from the
// workspace: one thread per quarter block.
__global__ void __launch_bounds__(256) act_quant_kernel(const GemvParams p) {
    pdl_launch_dependents();
    pdl_wait();   // X may come from the kernel before this one on the stream
    const int nb = (int)(p.K / 32);
    const int quarters = 4 * p.M * nb;
    const int idx = blockIdx.x * 256 + threadIdx.x;
    const bool on = idx < quarters;
    const int blk = on ? idx >> 2 : 0;
    quant_quarter(p, on, blk / nb, blk % nb, idx & 3, static_cast<uint8_t*>(p.act_image));
}

// Bytes of the activation image.
__host__ __device__ constexpr int64_t act_image_bytes(int64_t M, int64_t K) {
    return M * qa_row_stride(K) + M * (K / 32) * 16;
}

// Pulls the activation image into shared memory (one bulk copy) once the
// quantizer has finished; every thread returns after it has landed (or after
// the bounded wait gave up and reported GGUF_ERR_TIMEOUT).
__device__ __forceinline__ bool load_act_image(const GemvParams& p, const Shared& sh, uint64_t* bar) {
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t bytes = (uint32_t)act_image_bytes(p.M, p.K);
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s_u32(sh.qa, p.act_image, bytes, bar);
    }
    return mbar_wait(bar, 0, p.status);
}

// ------------------------------------------------------------------ per-lane activation slice
// The codes (NQ/4 16-byte pieces) and block entries (NE) a lane needs for one
// 128-value unit (NQ = 8, NE = 4) or one 32-value Q8_0 block (NQ = 2, NE = 1),
// held in registers (REG) or read from shared memory on demand.
template <int MT, bool REG, int NQ, int NE>
struct ActSlice {
    uint4 q[REG ? MT : 1][NQ];
    uint4 e[REG ? MT : 1][NE];
    uint32_t qa_base, ds_base, qa_row, ds_row;

    __device__ __forceinline__ void init(const Shared& sh, int k0, int nb, int m0 = 0) {
        qa_row = sh.qa_row;
        ds_row = 16u * (uint32_t)nb;
        qa_base = sh.qa + qa_pos((uint32_t)k0) + (uint32_t)m0 * qa_row;
        ds_base = sh.ds + 16u * (uint32_t)(k0 / 32) + (uint32_t)m0 * ds_row;
        if (REG) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int i = 0; i < NQ; ++i) q[REG ? m : 0][i] = lds128(qa_base + m * qa_row + 16 * i);
#pragma unroll
                for (int b = 0; b < NE; ++b) e[REG ? m : 0][b] = lds128(ds_base + m * ds_row + 16 * b);
            }
        }
    }
    // 16 codes: elements 16i .. 16i+15 of the unit, row m
    __device__ __forceinline__ uint4 codes(int m, int i) const {
        if (REG) return q[REG ? m : 0][i];
        return lds128(qa_base + m * qa_row + 16 * i);
    }
    __device__ __forceinline__ uint4 entry(int m, int b) const {
        if (REG) return e[REG ? m : 0][b];
        return lds128(ds_base + m * ds_row + 16 * b);
    }
};

__device__ __forceinline__ void dump_D(const GemvParams& p, int m, int64_t n, int j, int sub, int v) {
    p.dbg_D[((int64_t)m * p.N + n) * (p.K / sub) + j] = v;
}

// ------------------------------------------------------------------ Q4_K / Q5_K unit
// Fragment: the 16-byte header (d, dmin, 12 scale bytes), qh (Q5_K) and the 64
// qs bytes of half h.
template <int QT>
struct FragQ45 {
    uint4 hdr;
    uint4 qh[2];
    uint4 qs[4];
    // blk: shared address of the (16-byte aligned) block
    __device__ __forceinline__ void load(uint32_t blk, int h) {
        hdr = lds128(blk);
        if (QT == GGUF_Q5_K) { qh[0] = lds128(blk + 16); qh[1] = lds128(blk + 32); }
        const uint32_t q = blk + (QT == GGUF_Q5_K ? 48 : 16) + 64 * h;
#pragma unroll
        for (int i = 0; i < 4; ++i) qs[i] = lds128(q + 16 * i);
    }
};

// R rows of the same unit at once: every activation-code load is shared by the
// R rows' dot products.  f[r], acc[r], n[r], on[r]: fragment, accumulators,
// output row and validity of row r.
// m0: the first activation row the MT accumulators stand for (the accessor's
// row m is activation row m0 + m).
template <int QT, int MT, int R, class A, bool DUMP>
__device__ __forceinline__ void unit_q45k(const GemvParams& p, const FragQ45<QT>* const* f, const A& a, int kb,
                                          int h, float (*acc)[MT], const int64_t* n, const bool* on, int m0 = 0) {
    float d[R], dmin[R];
    uint32_t scw[R], mnw[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        d[r] = f16_bits_to_float(f[r]->hdr.x);
        dmin[r] = f16_bits_to_float(f[r]->hdr.x >> 16);
        // 6-bit scales (scw) and mins (mnw) of the sub-blocks 4h..4h+3, one per byte
        const uint32_t s0 = f[r]->hdr.y, s1 = f[r]->hdr.z, s2 = f[r]->hdr.w;
        scw[r] = h ? ((s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u)) : (s0 & 0x3F3F3F3Fu);
        mnw[r] = h ? (((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u)) : (s1 & 0x3F3F3F3Fu);
    }
    float accd[R][MT], accm[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) accd[r][m] = accm[r][m] = 0.f;
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        const int jj = 4 * h + 2 * pp;                 // sub-blocks jj (low nibbles) and jj+1 (high)
        uint32_t lo[R][8], hi[R][8];
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t q = comp(f[r]->qs[2 * pp + (i >> 2)], i);
                lo[r][i] = q & 0x0F0F0F0Fu;
                hi[r][i] = (q >> 4) & 0x0F0F0F0Fu;
                if (QT == GGUF_Q5_K) {
                    // bit jj (resp. jj+1) of every qh byte rotated to bit 4 of that byte
                    const uint32_t hb = comp(f[r]->qh[i >> 2], i);
                    lo[r][i] |= __funnelshift_l(hb, hb, (uint32_t)(4 - jj) & 31u) & 0x10101010u;
                    hi[r][i] |= __funnelshift_l(hb, hb, (uint32_t)(3 - jj) & 31u) & 0x10101010u;
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m0 + m < p.M) {
                const uint4 l0 = a.codes(m, 4 * pp), l1 = a.codes(m, 4 * pp + 1);
                const uint4 h0 = a.codes(m, 4 * pp + 2), h1 = a.codes(m, 4 * pp + 3);
                const uint4 e0 = a.entry(m, 2 * pp), e1 = a.entry(m, 2 * pp + 1);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    int D0a = 0, D0b = 0, D1a = 0, D1b = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        D0a = dp4a(lo[r][i], comp(l0, i), D0a);
                        D0b = dp4a(lo[r][4 + i], comp(l1, i), D0b);
                        D1a = dp4a(hi[r][i], comp(h0, i), D1a);
                        D1b = dp4a(hi[r][4 + i], comp(h1, i), D1b);
                    }
                    const int D0 = D0a + D0b, D1 = D1a + D1b;
                    const int sc0 = (scw[r] >> (16 * pp)) & 0xFF, sc1 = (scw[r] >> (16 * pp + 8)) & 0xFF;
                    const float mn0 = i2f((mnw[r] >> (16 * pp)) & 0xFF), mn1 = i2f((mnw[r] >> (16 * pp + 8)) & 0xFF);
                    accd[r][m] += __uint_as_float(e0.x) * i2f(sc0 * D0) + __uint_as_float(e1.x) * i2f(sc1 * D1);
                    accm[r][m] += mn0 * __uint_as_float(e0.y) + mn1 * __uint_as_float(e1.y);
                    if (DUMP && p.dbg_D && on[r]) {
                        dump_D(p, m0 + m, n[r], kb * 8 + jj, 32, D0);
                        dump_D(p, m0 + m, n[r], kb * 8 + jj + 1, 32, D1);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[r][m] += d[r] * accd[r][m] - dmin[r] * accm[r][m];
}

// ------------------------------------------------------------------ Q4_K / Q5_K unit, row-lane form
// Half H (values 128H .. 128H + 127) of super-block kb of one weight row, whose
// block starts at shared address blk, against MT activation rows.  The lanes of
// a warp hold different weight rows of the same unit, so the activation codes
// (row m at qa + m * qa_row: the unit's 128 codes) and block entries (row m at
// ds + m * ds_row: four entries of 16 bytes, of which {d_a, d_a * s} are read)
// sit at warp-uniform addresses and are served as broadcasts.  Each 64-value
// piece (sub-blocks j = 4H + 2pp and j + 1, the low and high nibbles of the
// same 32 qs bytes) is decoded once and dotted with every activation row, and
// only the qs bytes of the current piece are held, so four rows fit in the 64
// registers a lane has with two CTAs per SM.  With H a compile-time constant
// every shift amount is one too, and the shifts are written as multiplies
// (x << s = x * 2^s, x >> s = high half of x * 2^(32-s)), which the FMA pipe
// executes beside the ALU pipe that takes the masks.
__device__ __forceinline__ uint2 lds64(uint32_t a) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
    return v;
}
template <int S>
__device__ __forceinline__ uint32_t shift_fma(uint32_t x) {   // x << S for S >= 0, x >> -S for S < 0
    if constexpr (S >= 0) return x * (1u << S);
    else return __umulhi(x, 1u << (32 + S));
}

template <int QT, int MT, int H, bool DUMP>
__device__ __forceinline__ void unit_rl(const GemvParams& p, uint32_t blk, uint32_t qa, uint32_t qa_row, uint32_t ds,
                                        uint32_t ds_row, int kb, float (&acc)[MT], int64_t n) {
    const uint4 hdr = lds128(blk);
    const float d = f16_bits_to_float(hdr.x), dmin = f16_bits_to_float(hdr.x >> 16);
    // 6-bit scales and mins of sub-blocks 4H .. 4H + 3, one per byte (GGUF packing)
    const uint32_t scw = H ? ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u)) : (hdr.y & 0x3F3F3F3Fu);
    const uint32_t mnw = H ? (((hdr.w >> 4) & 0x0F0F0F0Fu) | ((hdr.z >> 2) & 0x30303030u)) : (hdr.z & 0x3F3F3F3Fu);
    uint4 qh0 = make_uint4(0, 0, 0, 0), qh1 = qh0;
    if constexpr (QT == GGUF_Q5_K) { qh0 = lds128(blk + 16); qh1 = lds128(blk + 32); }
    float accd[MT], accm[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) accd[m] = accm[m] = 0.f;
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        const uint32_t q = blk + (QT == GGUF_Q5_K ? 48u : 16u) + 64u * H + 32u * pp;
        const uint4 w0 = lds128(q), w1 = lds128(q + 16);
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w = comp(i < 4 ? w0 : w1, i);
            lo[i] = w & 0x0F0F0F0Fu;
            hi[i] = shift_fma<-4>(w) & 0x0F0F0F0Fu;
            if constexpr (QT == GGUF_Q5_K) {
                // bit jj (low nibbles) and jj + 1 (high nibbles) of each qh byte to bit 4
                const uint32_t hb = comp(i < 4 ? qh0 : qh1, i);
                if (pp == 0) {
                    lo[i] |= shift_fma<4 - 4 * H>(hb) & 0x10101010u;
                    hi[i] |= shift_fma<3 - 4 * H>(hb) & 0x10101010u;
                } else {
                    lo[i] |= shift_fma<2 - 4 * H>(hb) & 0x10101010u;
                    hi[i] |= shift_fma<1 - 4 * H>(hb) & 0x10101010u;
                }
            }
        }
        const int sc0 = (int)((scw >> (16 * pp)) & 0xFF), sc1 = (int)((scw >> (16 * pp + 8)) & 0xFF);
        const float mn0 = (float)((mnw >> (16 * pp)) & 0xFF), mn1 = (float)((mnw >> (16 * pp + 8)) & 0xFF);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < p.M) {
                const uint32_t c = qa + (uint32_t)m * qa_row + 64u * pp;
                int D0, D1;
                {
                    const uint4 l0 = lds128(c), l1 = lds128(c + 16);
                    int a = 0, b = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        a = dp4a(lo[i], comp(l0, i), a);
                        b = dp4a(lo[4 + i], comp(l1, i), b);
                    }
                    D0 = a + b;
                }
                {
                    const uint4 h0 = lds128(c + 32), h1 = lds128(c + 48);
                    int a = 0, b = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        a = dp4a(hi[i], comp(h0, i), a);
                        b = dp4a(hi[4 + i], comp(h1, i), b);
                    }
                    D1 = a + b;
                }
                const uint32_t e = ds + (uint32_t)m * ds_row + 32u * pp;
                const uint2 e0 = lds64(e), e1 = lds64(e + 16);
                accd[m] += __uint_as_float(e0.x) * i2f(sc0 * D0) + __uint_as_float(e1.x) * i2f(sc1 * D1);
                accm[m] += mn0 * __uint_as_float(e0.y) + mn1 * __uint_as_float(e1.y);
                if (DUMP && p.dbg_D) {
                    dump_D(p, m, n, kb * 8 + 4 * H + 2 * pp, 32, D0);
                    dump_D(p, m, n, kb * 8 + 4 * H + 2 * pp + 1, 32, D1);
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] += d * accd[m] - dmin * accm[m];
}

// ------------------------------------------------------------------ Q2_K / Q3_K unit
// Half h of a super-block (128 values; sub-blocks 8h .. 8h+7 of 16 values),
// its raw block staged in shared memory at `blk` (2-byte aligned).  Element
// r = 32j + 16p + l of the half is bits 2j..2j+1 of qs[32h + 16p + l]; its
// sub-block is 8h + 2j + p and its activation block is j (codes 16(2j+p) ..
// of the unit).  Q3_K's high bit (bit 4h + j of hmask[16p + l]) makes the code
// q2 + 4 hbit = q3 + 4 in 0..7, so a sub-block's dot of q3 is the unsigned
// dot less 4 times the sum of its 16 activation codes (the entry's s_lo or s_hi).
template <int QT, int MT, class A, bool DUMP>
__device__ __forceinline__ void unit_k23(const GemvParams& p, uint32_t blk, const A& a, int kb, int h,
                                         float (&acc)[MT], int64_t n) {
    constexpr bool Q2 = QT == GGUF_Q2_K;
    auto w32 = [&](uint32_t ad) { return lds16(ad) | (lds16(ad + 2) << 16); };   // word at a 2-byte aligned address
    uint32_t q[8];                                          // the half's 32 code bytes
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = w32(blk + (Q2 ? 16u : 32u) + 32u * (uint32_t)h + 4u * i);
    uint32_t hm[8];
    float d, dmin = 0.f;
    int sc[8], mn[8];                                       // sub-blocks 8h + t
    if constexpr (Q2) {
        d = f16_bits_to_float(lds16(blk + 80));
        dmin = f16_bits_to_float(lds16(blk + 82));
        const uint32_t s0 = w32(blk + 8u * (uint32_t)h), s1 = w32(blk + 8u * (uint32_t)h + 4u);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int b = (int)(((t < 4 ? s0 : s1) >> (8 * (t & 3))) & 0xFF);
            sc[t] = b & 15;
            mn[t] = b >> 4;
        }
    } else {
        d = f16_bits_to_float(lds16(blk + 108));
#pragma unroll
        for (int i = 0; i < 8; ++i) hm[i] = w32(blk + 4u * i);
        const uint32_t s0 = w32(blk + 96), s1 = w32(blk + 100), s2 = w32(blk + 104);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            // scale 8h + t: low 4 bits from byte t (low nibble in half 0, high in half 1),
            // top 2 bits from byte 8 + t%4, bits 2((8h + t)/4) = 4h + 2(t/4)
            const uint32_t byte = ((t < 4 ? s0 : s1) >> (8 * (t & 3))) & 0xFF;
            const uint32_t low = h ? (byte >> 4) : (byte & 15);
            const uint32_t top = ((s2 >> (8 * (t & 3))) >> (4 * h + 2 * (t >> 2))) & 3;
            sc[t] = (int)(low | (top << 4)) - 32;
            mn[t] = 0;
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < p.M) {
            float u = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 en = a.entry(m, j);
                int S = 0, Mn = 0;
#pragma unroll
                for (int pp = 0; pp < 2; ++pp) {
                    const uint4 codes = a.codes(m, 2 * j + pp);
                    const int s16 = (int)(pp ? en.w : en.z);
                    int D = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint32_t v = (q[4 * pp + i] >> (2 * j)) & 0x03030303u;
                        if constexpr (!Q2) v |= ((hm[4 * pp + i] >> (4 * h + j)) & 0x01010101u) << 2;
                        D = dp4a(v, comp(codes, i), D);
                    }
                    if constexpr (!Q2) D -= 4 * s16;
                    S += sc[2 * j + pp] * D;
                    Mn += mn[2 * j + pp] * s16;
                    if (DUMP && p.dbg_D) dump_D(p, m, n, kb * 16 + 8 * h + 2 * j + pp, 16, D);
                }
                u += __uint_as_float(en.x) * (d * i2f(S) - dmin * i2f(Mn));
            }
            acc[m] += u;
        }
    }
}

// ------------------------------------------------------------------ Q6_K unit
struct FragQ6 {
    uint4 ql[4];   // 64 bytes of ql for half h
    uint4 qh[2];   // 32 bytes of qh for half h
    uint2 sc;      // 8 scales for half h
    uint32_t d;    // f16 bits
};

template <int MT, int R, class A, bool DUMP>
__device__ __forceinline__ void unit_q6k(const GemvParams& p, const FragQ6* const* f, const A& a, int kb, int h,
                                         float (*acc)[MT], const int64_t* n, const bool* on) {
    float d[R];
    int sc[R][8];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        d[r] = f16_bits_to_float(f[r]->d);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            sc[r][t] = (int)(int8_t)((f[r]->sc.x >> (8 * t)) & 0xFF);
            sc[r][4 + t] = (int)(int8_t)((f[r]->sc.y >> (8 * t)) & 0xFF);
        }
    }
    int S[R][MT][4];   // per activation block b (0..3 of the unit): sum of sc_t * D_t over its two sub-blocks
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int m = 0; m < MT; ++m) S[r][m][0] = S[r][m][1] = S[r][m][2] = S[r][m][3] = 0;
#pragma unroll
    for (int gp = 0; gp < 2; ++gp) {
        // gp = 0: groups g = 0 (low nibbles) and g = 2 (high nibbles) of ql[0..31]
        // gp = 1: groups g = 1 and g = 3 of ql[32..63]
        uint32_t qlo[R][8], qhi[R][8];
#pragma unroll
        for (int r = 0; r < R; ++r) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t X = comp(f[r]->ql[2 * gp + (i >> 2)], i), H = comp(f[r]->qh[i >> 2], i);
                qlo[r][i] = (X & 0x0F0F0F0Fu) | ((H << (4 - 2 * gp)) & 0x30303030u);
                qhi[r][i] = ((X >> 4) & 0x0F0F0F0Fu) | ((H >> (2 * gp)) & 0x30303030u);
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < p.M) {
                const uint4 l0 = a.codes(m, 2 * gp), l1 = a.codes(m, 2 * gp + 1);
                const uint4 h0 = a.codes(m, 4 + 2 * gp), h1 = a.codes(m, 5 + 2 * gp);
                const uint4 el = a.entry(m, gp), eh = a.entry(m, 2 + gp);
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    int Dl0 = 0, Dl1 = 0, Dh0 = 0, Dh1 = 0;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        Dl0 = dp4a(qlo[r][i], comp(l0, i), Dl0);
                        Dl1 = dp4a(qlo[r][4 + i], comp(l1, i), Dl1);
                        Dh0 = dp4a(qhi[r][i], comp(h0, i), Dh0);
                        Dh1 = dp4a(qhi[r][4 + i], comp(h1, i), Dh1);
                    }
                    // dots of (q6 - 32): subtract 32 * (sum of the 16 activation codes)
                    Dl0 -= 32 * (int)el.z; Dl1 -= 32 * (int)el.w;
                    Dh0 -= 32 * (int)eh.z; Dh1 -= 32 * (int)eh.w;
                    S[r][m][gp] += sc[r][2 * gp] * Dl0 + sc[r][2 * gp + 1] * Dl1;
                    S[r][m][2 + gp] += sc[r][4 + 2 * gp] * Dh0 + sc[r][5 + 2 * gp] * Dh1;
                    if (DUMP && p.dbg_D && on[r]) {
                        dump_D(p, m, n[r], kb * 16 + 8 * h + 2 * gp, 16, Dl0);
                        dump_D(p, m, n[r], kb * 16 + 8 * h + 2 * gp + 1, 16, Dl1);
                        dump_D(p, m, n[r], kb * 16 + 8 * h + 4 + 2 * gp, 16, Dh0);
                        dump_D(p, m, n[r], kb * 16 + 8 * h + 5 + 2 * gp, 16, Dh1);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < p.M) {
            float da[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) da[b] = __uint_as_float(a.entry(m, b).x);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float u = 0.f;
#pragma unroll
                for (int b = 0; b < 4; ++b) u += da[b] * i2f(S[r][m][b]);
                acc[r][m] += d[r] * u;
            }
        }
    }
}

// ------------------------------------------------------------------ Q8_0 unit (from shared memory)
template <int MT, class A, bool DUMP>
__device__ __forceinline__ void unit_q8_0(const GemvParams& p, uint32_t blk, const A& a, int b, float acc[MT],
                                          int64_t n) {
    const float d = f16_bits_to_float(lds16(blk));
    uint32_t q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = lds16(blk + 2 + 4 * i) | (lds16(blk + 4 + 4 * i) << 16);
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < p.M) {
            const uint4 c0 = a.codes(m, 0), c1 = a.codes(m, 1);
            int Da = 0, Db = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                Da = dp4a(q[i], comp(c0, i), Da);
                Db = dp4a(q[4 + i], comp(c1, i), Db);
            }
            const int D = Da + Db;
            acc[m] += d * (__uint_as_float(a.entry(m, 0).x) * i2f(D));
            if (DUMP && p.dbg_D) dump_D(p, m, n, b, 32, D);
        }
    }
}

// ------------------------------------------------------------------ Q4_0 / Q4_1 / Q5_0 / Q5_1 unit (from shared memory)
// One 32-value block at the 2-byte-aligned shared address blk.  The codes are
// dotted unsigned (0..15, or 0..31 with the fifth bit); the formats' zero
// point and min are applied through the activation block's code sum s:
//   Q4_0: D = sum (q - 8) qa = sum q qa - 8 s      y += d * d_a * D
//   Q5_0: D = sum (q5 - 16) qa = sum q5 qa - 16 s  y += d * d_a * D
//   Q4_1 / Q5_1: D = sum q qa                      y += d * d_a * D + m * d_a * s
// Four bits of the qh word are spread to bit 4 of four bytes with one multiply
// (b * 0x00204081 puts bit i of b at bit 8i + i ... then a mask).
__device__ __forceinline__ uint32_t spread4_to_bit4(uint32_t b) {
    return ((b & 0xFu) * 0x00204081u & 0x01010101u) << 4;
}
template <int QT, int MT, class A, bool DUMP>
__device__ __forceinline__ void unit_b32(const GemvParams& p, uint32_t blk, const A& a, int b, float acc[MT],
                                         int64_t n) {
    const float d = f16_bits_to_float(lds16(blk));
    const float mval = b32_has_min(QT) ? f16_bits_to_float(lds16(blk + 2)) : 0.f;
    const uint32_t qs = blk + b32_qs_offset(QT);
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t w = lds16(qs + 4 * i) | (lds16(qs + 4 * i + 2) << 16);
        lo[i] = w & 0x0F0F0F0Fu;
        hi[i] = (w >> 4) & 0x0F0F0F0Fu;
    }
    if constexpr (b32_has_qh(QT)) {
        const uint32_t qh = lds16(qs - 4) | (lds16(qs - 2) << 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] |= spread4_to_bit4(qh >> (4 * i));
            hi[i] |= spread4_to_bit4(qh >> (16 + 4 * i));
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < p.M) {
            const uint4 c0 = a.codes(m, 0), c1 = a.codes(m, 1);
            int Da = 0, Db = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                Da = dp4a(lo[i], comp(c0, i), Da);
                Db = dp4a(hi[i], comp(c1, i), Db);
            }
            const uint4 e = a.entry(m, 0);
            int D = Da + Db;
            if (b32_zero_point(QT)) D -= b32_zero_point(QT) * (int)(e.z + e.w);
            acc[m] += d * (__uint_as_float(e.x) * i2f(D));
            if (b32_has_min(QT)) acc[m] += mval * __uint_as_float(e.y);
            if (DUMP && p.dbg_D) dump_D(p, m, n, b, 32, D);
        }
    }
}

// Q6_K fragment of half h from a 2-byte-aligned raw block in shared memory.
__device__ __forceinline__ void frag_q6_from_smem(FragQ6& f, uint32_t blk, int h) {
    auto w32 = [&](uint32_t a) { return lds16(a) | (lds16(a + 2) << 16); };
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t q = blk + 64 * h + 16 * i;
        f.ql[i] = make_uint4(w32(q), w32(q + 4), w32(q + 8), w32(q + 12));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t q = blk + 128 + 32 * h + 16 * i;
        f.qh[i] = make_uint4(w32(q), w32(q + 4), w32(q + 8), w32(q + 12));
    }
    f.sc = make_uint2(w32(blk + 192 + 8 * h), w32(blk + 196 + 8 * h));
    f.d = lds16(blk + 208);
}

// Q6_K fragment of half h from the plane pieces staged in shared memory.
__device__ __forceinline__ void frag_q6_from_planes(FragQ6& f, uint32_t ql, uint32_t qh, uint32_t sc, uint32_t d,
                                                    int h) {
#pragma unroll
    for (int i = 0; i < 4; ++i) f.ql[i] = lds128(ql + 64 * h + 16 * i);
    f.qh[0] = lds128(qh + 32 * h);
    f.qh[1] = lds128(qh + 32 * h + 16);
    f.sc = make_uint2(lds32(sc + 8 * h), lds32(sc + 8 * h + 4));
    f.d = lds16(d);
}


// Stages global bytes [lo, hi) of the weight buffer (total bytes) in shared
// memory at dst, starting from the 16-byte boundary at or below lo: byte x
// lands at dst + (x - (lo & ~15)).  The 16-byte-granular body goes as one 1-D
// bulk (TMA) copy that completes its bytes on `bar`; the few bytes past the
// last whole 16-byte piece of the buffer are stored by this thread.  Returns
// the bulk byte count (the caller adds it to the barrier's expected bytes
// before issuing).  Called by one lane.
struct BulkPiece {
    uint32_t dst;
    const uint8_t* src;
    uint32_t bytes;
};
__device__ __forceinline__ BulkPiece stage_range(uint32_t dst, const uint8_t* w, int64_t lo, int64_t hi,
                                                 int64_t total) {
    const int64_t a0 = lo & ~int64_t(15);
    const int64_t e = min((hi + 15) & ~int64_t(15), total & ~int64_t(15));
    for (int64_t x = max(e, a0); x < min(hi, total); ++x)
        asm volatile("st.shared.u8 [%0], %1;" ::"r"(dst + (uint32_t)(x - a0)), "h"((unsigned short)w[x]));
    return BulkPiece{dst, w + a0, e > a0 ? (uint32_t)(e - a0) : 0u};
}

// ------------------------------------------------------------------ the kernel
// Row groups: a warp pass covers P rows (P = 32 / U when a row has U < 32
// units, else 1); groups are dealt to warps round-robin.  Each warp stages its
// groups through a ring of R slots of p.stage_bytes in shared memory.
template <int QT, int MT, int LAYOUT, bool REG, bool DUMP, bool ROUTED = false>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const GemvParams p) {
    constexpr int NT = kThreads, NW = NT / 32;
    constexpr bool PLANES = QT == GGUF_Q6_K && LAYOUT == GGUF_LAYOUT_Q6K_PLANES;
    constexpr bool B32 = block32(QT);                 // 32-value blocks: a unit is one block
    constexpr int NQ = B32 ? 2 : 8, NE = B32 ? 1 : 4;
    constexpr int UV = B32 ? 32 : 128;                // values per unit
    constexpr int bb = block_bytes(QT);
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = (int)(p.K / 32);
    static_assert(!ROUTED || (MT == 1 && !DUMP), "routed rows: one activation row, no dumps");
    // routed mode: this grid row's expert (a row without one is left untouched),
    // its weights, and the output row it writes
    const uint8_t* wsrc = p.w;
    int64_t out_off = 0, arow = 0;
    if constexpr (ROUTED) {
        const int r = (int)blockIdx.y;
        const int e = p.ids[r];
        if (e < 0 || e >= p.n_expert) return;   // uniform exit before any shared state exists
        wsrc = p.w + (int64_t)e * p.N * p.rb;
        out_off = (int64_t)r * p.N;
        arow = r / p.route_div;
    }
    Shared sh;
    sh.qa_row = (uint32_t)qa_row_stride(p.K);
    sh.qa = smem_u32(smem_raw);
    sh.ds = sh.qa + (uint32_t)p.M * sh.qa_row;
    sh.stage = sh.ds + 16u * (uint32_t)(p.M * nb);

    const int64_t row0 = (int64_t)blockIdx.x * p.rows_per_cta;
    const int64_t row_end = min(p.N, row0 + p.rows_per_cta);
    const int U = (int)(p.K / UV);                  // units per row
    const int seg = U < 32 ? U : 32;
    const int P = U < 32 ? 32 / U : 1;              // rows per warp pass
    const int64_t KB = p.K / 256, nblk = p.N * KB, total = p.N * p.rb;
    const int u0 = U < 32 ? lane % U : lane;        // this lane's first unit
    const int sub_row = U < 32 ? lane / U : 0;
    const bool lane_on = U >= 32 || lane < P * U;
    const int groups = row0 < row_end ? (int)ceil_div(row_end - row0, P) : 0;
    const int R = p.stages;
    const uint32_t ring = sh.stage + (uint32_t)(warp * R) * (uint32_t)p.stage_bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + (sh.stage - sh.qa) + (size_t)NW * R * p.stage_bytes) +
                     warp * R;
    const int64_t pb = (int64_t)P * KB;             // blocks per group (planes)
    if (lane == 0) {
        for (int i = 0; i < R; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // slot layout: raw bytes of the group's rows; or the four plane pieces
    // QL | QH | SC | D of its pb blocks (D from its 16-byte boundary)
    auto issue = [&](int g, int slot) {
        if (lane != 0) return;
        const int64_t r_begin = row0 + (int64_t)g * P;
        const int64_t rows = min((int64_t)P, row_end - r_begin);
        const uint32_t dst = ring + (uint32_t)slot * (uint32_t)p.stage_bytes;
        BulkPiece pc[4];
        int np = 0;
        if (PLANES) {
            const int64_t b0 = r_begin * KB, cb = rows * KB;
            pc[np++] = stage_range(dst, p.w, 128 * b0, 128 * (b0 + cb), total);
            pc[np++] = stage_range(dst + (uint32_t)(128 * pb), p.w, 128 * nblk + 64 * b0, 128 * nblk + 64 * (b0 + cb), total);
            pc[np++] = stage_range(dst + (uint32_t)(192 * pb), p.w, 192 * nblk + 16 * b0, 192 * nblk + 16 * (b0 + cb), total);
            pc[np++] = stage_range(dst + (uint32_t)(208 * pb), p.w, 208 * nblk + 2 * b0, 208 * nblk + 2 * (b0 + cb), total);
        } else {
            pc[np++] = stage_range(dst, wsrc, r_begin * p.rb, (r_begin + rows) * p.rb, total);
        }
        uint32_t tx = 0;
        for (int i = 0; i < np; ++i) tx += pc[i].bytes;
        // the slot was last read through the generic proxy: order those reads
        // before the bulk copy's writes
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&bars[slot], tx);
        for (int i = 0; i < np; ++i)
            if (pc[i].bytes) bulk_g2s_u32(pc[i].dst, pc[i].src, pc[i].bytes, &bars[slot]);
    };

    // 1. request the first R groups of this warp
    for (int i = 0; i < R && warp + i * NW < groups; ++i) issue(warp + i * NW, i);
    pdl_launch_dependents();

    // 2. activation prologue, once the producer of X has finished
    pdl_wait();
    if constexpr (ROUTED) {
        // this row's codes and block entries out of the image of img_rows rows
        uint64_t* bar = bars + (NW - warp) * R;
        if (threadIdx.x == 0) {
            mbar_init(bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            const uint8_t* img = static_cast<const uint8_t*>(p.act_image);
            const uint32_t cb = sh.qa_row, eb = 16u * (uint32_t)nb;
            mbar_arrive_expect_tx(bar, cb + eb);
            bulk_g2s_u32(sh.qa, img + arow * cb, cb, bar);
            bulk_g2s_u32(sh.ds, img + p.img_rows * cb + arow * eb, eb, bar);
        }
        mbar_wait(bar, 0, p.status);
    } else {
        load_act_image(p, sh, bars + (NW - warp) * R);   // the barrier after the ring's
    }
    __syncthreads();
    if (DUMP && blockIdx.x == 0) {
        for (int64_t i = tid; i < (int64_t)p.M * p.K; i += NT) {
            const uint32_t a = sh.qa + (uint32_t)(i / p.K) * sh.qa_row + qa_pos((uint32_t)(i % p.K));
            if (p.dbg_qa) p.dbg_qa[i] = (int8_t)(lds32(a & ~3u) >> (8 * (a & 3)));
        }
        for (int i = tid; i < p.M * nb; i += NT) {
            const uint4 e = lds128(sh.ds + 16u * i);
            if (p.dbg_da) p.dbg_da[i] = __uint_as_float(e.x);
            if (p.dbg_s) p.dbg_s[i] = (int32_t)(e.z + e.w);
        }
    }
    ActSlice<MT, REG, NQ, NE> act;   // this lane's slice (its only unit when U <= 32)
    act.init(sh, UV * u0, nb);
    const bool single_unit = U <= 32;

    // 3. rows
    const int seg_end = (lane / seg) * seg + seg;   // one segment of lanes per row
    const bool head = lane_on && (lane % seg) == 0;
    const uint32_t rb32 = (uint32_t)p.rb;
    int slot = 0;
    uint32_t phase = 0;   // bit i: parity of the next completion of slot i
    for (int g = warp; g < groups; g += NW) {
        const int ok = mbar_wait(&bars[slot], (phase >> slot) & 1u, p.status) ? 1 : 0;
        phase ^= 1u << slot;
        if (!__all_sync(0xffffffffu, ok)) break;
        const uint32_t sbase = ring + (uint32_t)slot * (uint32_t)p.stage_bytes;
        const int64_t r_begin = row0 + (int64_t)g * P;
        const int64_t n = r_begin + sub_row;
        const bool valid = lane_on && n < row_end;
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        if (valid) {
            const uint32_t rowp = sbase + (uint32_t)((uint64_t)r_begin * p.rb & 15) + (uint32_t)sub_row * rb32;
            for (int u = u0; u < U; u += (U < 32 ? U : 32)) {
                const int kb = u >> 1, h = u & 1;
                ActSlice<MT, false, NQ, NE> as;
                if (!single_unit) as.init(sh, UV * u, nb);
                if constexpr (QT == GGUF_Q8_0) {
                    if (single_unit) unit_q8_0<MT, decltype(act), DUMP>(p, rowp + 34u * u, act, u, acc, n);
                    else unit_q8_0<MT, decltype(as), DUMP>(p, rowp + 34u * u, as, u, acc, n);
                } else if constexpr (B32) {
                    if (single_unit) unit_b32<QT, MT, decltype(act), DUMP>(p, rowp + (uint32_t)bb * u, act, u, acc, n);
                    else unit_b32<QT, MT, decltype(as), DUMP>(p, rowp + (uint32_t)bb * u, as, u, acc, n);
                } else if constexpr (k23(QT)) {
                    if (single_unit) unit_k23<QT, MT, decltype(act), DUMP>(p, rowp + (uint32_t)bb * kb, act, kb, h, acc, n);
                    else unit_k23<QT, MT, decltype(as), DUMP>(p, rowp + (uint32_t)bb * kb, as, kb, h, acc, n);
                } else if constexpr (QT == GGUF_Q6_K) {
                    FragQ6 f;
                    if constexpr (PLANES) {
                        const uint32_t bi = (uint32_t)(sub_row * KB + kb);
                        const uint32_t dq = sbase + (uint32_t)(208 * pb) + (uint32_t)(((r_begin * KB) * 2) & 15);
                        frag_q6_from_planes(f, sbase + 128u * bi, sbase + (uint32_t)(128 * pb) + 64u * bi,
                                            sbase + (uint32_t)(192 * pb) + 16u * bi, dq + 2u * bi, h);
                    } else {
                        frag_q6_from_smem(f, rowp + 210u * kb, h);
                    }
                    const FragQ6* fp1[1] = {&f};
                    const int64_t n1[1] = {n};
                    const bool on1[1] = {true};
                    if (single_unit) unit_q6k<MT, 1, decltype(act), DUMP>(p, fp1, act, kb, h, &acc, n1, on1);
                    else unit_q6k<MT, 1, decltype(as), DUMP>(p, fp1, as, kb, h, &acc, n1, on1);
                } else {
                    FragQ45<QT> f;
                    f.load(rowp + (uint32_t)(bb * kb), h);
                    const FragQ45<QT>* fp1[1] = {&f};
                    const int64_t n1[1] = {n};
                    const bool on1[1] = {true};
                    if (single_unit) unit_q45k<QT, MT, 1, decltype(act), DUMP>(p, fp1, act, kb, h, &acc, n1, on1);
                    else unit_q45k<QT, MT, 1, decltype(as), DUMP>(p, fp1, as, kb, h, &acc, n1, on1);
                }
            }
        }
        // refill this slot with the group R passes ahead, once every lane is done with it
        __syncwarp();
        if (g + R * NW < groups) issue(g + R * NW, slot);
        if (++slot == R) slot = 0;
        if (seg == 32) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
            }
        } else {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float t = __shfl_down_sync(0xffffffffu, acc[m], o);
                    if (lane + o < seg_end) acc[m] += t;
                }
            }
        }
        if (head && valid) {
            for (int m = 0; m < p.M && m < MT; ++m) {
                float v = acc[m];
                if (p.residual) v += load_act(p.residual, p.ydt, out_off + (int64_t)m * p.N + n);
                store_out(p.y, p.ydt, out_off + (int64_t)m * p.N + n, v);
            }
        }
    }
}

// ------------------------------------------------------------------ direct-load kernel
// For the layouts whose unit fields are 16-byte aligned (Q4_K, Q5_K blocks and
// the Q6_K planes): each lane fetches exactly its unit's bytes with 128-bit
// loads straight into registers, one (row, unit) item ahead of the one it
// computes; the first item is requested before waiting on the producer of X.
__device__ __forceinline__ uint4 ldg128(const uint8_t* p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ uint2 ldg64(const uint8_t* p) {
    uint2 v;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg16(const uint8_t* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

template <int QT>
__device__ __forceinline__ void load_global(FragQ45<QT>& f, const uint8_t* blk, int h) {
    f.hdr = ldg128(blk);
    if (QT == GGUF_Q5_K) { f.qh[0] = ldg128(blk + 16); f.qh[1] = ldg128(blk + 32); }
    const uint8_t* q = blk + (QT == GGUF_Q5_K ? 48 : 16) + 64 * h;
#pragma unroll
    for (int i = 0; i < 4; ++i) f.qs[i] = ldg128(q + 16 * i);
}

__device__ __forceinline__ void load_global_planes(FragQ6& f, const uint8_t* w, int64_t nblk, int64_t b, int h) {
    const uint8_t* ql = w + 128 * b + 64 * h;
    const uint8_t* qh = w + 128 * nblk + 64 * b + 32 * h;
#pragma unroll
    for (int i = 0; i < 4; ++i) f.ql[i] = ldg128(ql + 16 * i);
    f.qh[0] = ldg128(qh);
    f.qh[1] = ldg128(qh + 16);
    f.sc = ldg64(w + 192 * nblk + 16 * b + 8 * h);
    f.d = ldg16(w + 208 * nblk + 2 * b);
}

// One CTA per SM: 16 warps for M = 1, fewer as the per-lane state grows with M.
__host__ __device__ constexpr int direct_threads(int mt) { return mt == 1 ? 512 : mt == 2 ? 384 : 256; }

template <int QT, int MT, bool DUMP>
__global__ void __launch_bounds__(direct_threads(MT), 1) gemv_direct_kernel(const GemvParams p) {
    constexpr int NT = direct_threads(MT), NW = NT / 32;
    constexpr int bb = QT == GGUF_Q4_K ? 144 : QT == GGUF_Q5_K ? 176 : 210;
    using Frag = typename std::conditional<QT == GGUF_Q6_K, FragQ6, FragQ45<QT == GGUF_Q6_K ? GGUF_Q4_K : QT>>::type;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = (int)(p.K / 32);
    Shared sh;
    sh.qa_row = (uint32_t)qa_row_stride(p.K);
    sh.qa = smem_u32(smem_raw);
    sh.ds = sh.qa + (uint32_t)p.M * sh.qa_row;
    sh.stage = 0;

    const int64_t row0 = (int64_t)blockIdx.x * p.rows_per_cta;
    const int64_t row_end = min(p.N, row0 + p.rows_per_cta);
    const int U = (int)(p.K / 128);                 // units per row
    const int seg = U < 32 ? U : 32;
    const int P = U < 32 ? 32 / U : 1;              // rows per warp pass
    const int ustep = U < 32 ? U : 32;
    const int64_t KB = p.K / 256, nblk = p.N * KB;
    const int u0 = U < 32 ? lane % U : lane;
    const int sub_row = U < 32 ? lane / U : 0;
    const bool lane_on = U >= 32 || lane < P * U;
    const int groups = row0 < row_end ? (int)ceil_div(row_end - row0, P) : 0;

    Frag f0, f1;   // two-slot ring: the item being computed and the next one
    auto fetch = [&](Frag& f, int g, int u) {
        const int64_t n = row0 + (int64_t)g * P + sub_row;
        if (!lane_on || n >= row_end) return;
        const int kb = u >> 1, h = u & 1;
        if constexpr (QT == GGUF_Q6_K) load_global_planes(f, p.w, nblk, n * KB + kb, h);
        else load_global<QT>(f, p.w + n * p.rb + (int64_t)kb * bb, h);
    };
    // items (row group g, unit u) of this lane in order
    auto advance = [&](int g, int u, int& gn, int& un) {
        un = u + ustep;
        gn = g;
        if (un >= U) { un = u0; gn = g + NW; }
    };
    int g = warp, u = u0;
    {
        int g1, u1;
        advance(g, u, g1, u1);
        if (g < groups) fetch(f0, g, u);
        if (g1 < groups) fetch(f1, g1, u1);
    }
    pdl_launch_dependents();

    pdl_wait();
    // the CTA's residual values: one round trip for all of them, under the
    // image copy (shared memory after the image barrier)
    float* res = reinterpret_cast<float*>(smem_raw + (sh.ds - sh.qa) + 16 * p.M * nb + 16);
    const int nrows = row0 < row_end ? (int)(row_end - row0) : 0;
    float res0 = 0.f;
    if (p.residual && tid < p.M * nrows)
        res0 = load_act(p.residual, p.ydt, (int64_t)(tid / nrows) * p.N + row0 + tid % nrows);
    load_act_image(p, sh, reinterpret_cast<uint64_t*>(smem_raw + (sh.ds - sh.qa) + 16 * p.M * nb));
    if (p.residual) {
        if (tid < p.M * nrows) res[(tid / nrows) * p.rows_per_cta + tid % nrows] = res0;
        for (int i = tid + NT; i < p.M * nrows; i += NT)
            res[(i / nrows) * p.rows_per_cta + i % nrows] =
                load_act(p.residual, p.ydt, (int64_t)(i / nrows) * p.N + row0 + i % nrows);
    }
    __syncthreads();
    if (DUMP && blockIdx.x == 0) {
        for (int64_t i = tid; i < (int64_t)p.M * p.K; i += NT) {
            const uint32_t a = sh.qa + (uint32_t)(i / p.K) * sh.qa_row + qa_pos((uint32_t)(i % p.K));
            if (p.dbg_qa) p.dbg_qa[i] = (int8_t)(lds32(a & ~3u) >> (8 * (a & 3)));
        }
        for (int i = tid; i < p.M * nb; i += NT) {
            const uint4 e = lds128(sh.ds + 16u * i);
            if (p.dbg_da) p.dbg_da[i] = __uint_as_float(e.x);
            if (p.dbg_s) p.dbg_s[i] = (int32_t)(e.z + e.w);
        }
    }
    const bool single_unit = U <= 32;
    ActSlice<MT, false, 8, 4> fixed;
    fixed.init(sh, 128 * u0, nb);
    const int seg_end = (lane / seg) * seg + seg;
    const bool head = lane_on && (lane % seg) == 0;

    using Act = ActSlice<MT, false, 8, 4>;
    // reduction of one row's lane partials and the fused residual store
    auto finish_row = [&](float (&acc)[MT], int64_t n, bool valid) {
        if (seg == 32) {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
            }
        } else {
#pragma unroll
            for (int m = 0; m < MT; ++m) {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float t = __shfl_down_sync(0xffffffffu, acc[m], o);
                    if (lane + o < seg_end) acc[m] += t;
                }
            }
        }
        if (head && valid) {
            for (int m = 0; m < p.M && m < MT; ++m) {
                float v = acc[m];
                if (p.residual) v += res[m * p.rows_per_cta + (n - row0)];
                store_out(p.y, p.ydt, (int64_t)m * p.N + n, v);
            }
        }
    };

    if (single_unit) {
        // each lane has one unit per row: take the warp's rows two at a time, so
        // that every activation-code load serves both rows
        const int kb = u0 >> 1, h = u0 & 1;
        for (; g < groups; g += 2 * NW) {
            const int64_t n0r = row0 + (int64_t)g * P + sub_row, n1r = n0r + (int64_t)NW * P;
            const bool v0 = lane_on && n0r < row_end;
            const bool v1 = lane_on && g + NW < groups && n1r < row_end;
            float acc[2][MT];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
            const Frag* fr[2] = {&f0, &f1};
            const int64_t nn[2] = {n0r, n1r};
            const bool on[2] = {v0, v1};
            if constexpr (QT == GGUF_Q6_K) unit_q6k<MT, 2, Act, DUMP>(p, fr, fixed, kb, h, acc, nn, on);
            else unit_q45k<QT, MT, 2, Act, DUMP>(p, fr, fixed, kb, h, acc, nn, on);
            if (g + 2 * NW < groups) fetch(f0, g + 2 * NW, u0);
            if (g + 3 * NW < groups) fetch(f1, g + 3 * NW, u0);
            finish_row(acc[0], n0r, v0);
            finish_row(acc[1], n1r, v1);
        }
        return;
    }

    // long rows (several units per lane): one item at a time, the ring refilled
    // with the item two ahead
    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.f;
    auto step = [&](Frag& f) -> bool {
        if (g >= groups) return false;
        int gn, un, g2, u2;
        advance(g, u, gn, un);
        advance(gn, un, g2, u2);
        const int64_t n = row0 + (int64_t)g * P + sub_row;
        const bool valid = lane_on && n < row_end;
        if (valid) {
            Act moving;
            moving.init(sh, 128 * u, nb);
            const int kb = u >> 1, h = u & 1;
            const Frag* fr[1] = {&f};
            const int64_t nn[1] = {n};
            const bool on[1] = {true};
            float(*a1)[MT] = reinterpret_cast<float(*)[MT]>(&acc);
            if constexpr (QT == GGUF_Q6_K) unit_q6k<MT, 1, Act, DUMP>(p, fr, moving, kb, h, a1, nn, on);
            else unit_q45k<QT, MT, 1, Act, DUMP>(p, fr, moving, kb, h, a1, nn, on);
        }
        if (g2 < groups) fetch(f, g2, u2);
        if (gn != g) {
            finish_row(acc, n, valid);
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        }
        g = gn;
        u = un;
        return true;
    };
    while (step(f0) && step(f1)) {
    }
}

// ------------------------------------------------------------------ tile kernel
// Q4_K / Q5_K blocks, for shapes where a CTA's share of W and its activation
// image fit in half of an SM's shared memory.  Two CTAs then share an SM: the
// CTA of the next call on the stream (programmatic dependent launch) becomes
// resident while this call computes, and its first act is to request all of
// its weight bytes with bulk copies -- so the next call's weight stream runs
// under this call's compute and a chain of calls is bound by HBM rather than
// by per-call latency.  After its dependency wait the CTA quantizes the
// activation row itself (one kernel and one wait per call) and reads its
// residual values once into shared memory.
// One mbarrier per group of P rows (the rows a warp pass covers); warps take
// groups round-robin; a lane's unit is the same for every row.
// warps per CTA -- 16 at M = 1 (more rows in flight; the registers allow it),
// else 8 -- and row groups per warp iteration (one: measured faster at M = 1
// than 8 warps taking two rows at a time)
__host__ __device__ constexpr int tile_warps(int mt) { return mt == 1 ? 16 : 8; }
__host__ __device__ constexpr int tile_rows(int mt) { return 1; }

// Shared-memory layout of the tile kernel (byte offsets).
struct TileLayout {
    int64_t img, res, bars, total;
};
__host__ __device__ inline TileLayout tile_layout(int64_t M, int64_t K, int64_t rows_per_cta, int64_t rb) {
    const int64_t U = K / 128;
    const int64_t P = U < 32 ? 32 / U : 1;
    TileLayout L;
    L.img = ceil_div(rows_per_cta * rb, 128) * 128;
    L.res = L.img + ceil_div(act_image_bytes(M, K), 16) * 16;
    L.bars = L.res + ceil_div(4 * M * rows_per_cta, 16) * 16;
    L.total = L.bars + 8 * ceil_div(rows_per_cta, P);
    return L;
}

template <int QT, int MT, bool DUMP>
__global__ void __launch_bounds__(tile_warps(MT) * 32, 2) gemv_tile_kernel(const GemvParams p) {
    constexpr int NW = tile_warps(MT), NT = NW * 32;
    constexpr int bb = QT == GGUF_Q4_K ? 144 : 176;
    constexpr int TR = tile_rows(MT);
    constexpr bool AREG = false;     // activation codes read from shared memory
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row0 = (int64_t)blockIdx.x * p.rows_per_cta;
    const int rows = (int)min(p.rows_per_cta, p.N - row0);
    const int klen = (int)p.K;
    const int kb0 = 0;
    const int nbs = klen / 32;                    // activation blocks
    const int U = klen / 128;                     // units per row
    const int P = U < 32 ? 32 / U : 1;            // rows per warp pass
    const int ngroups = (rows + P - 1) / P;
    const uint32_t sb = (uint32_t)p.rb;           // bytes of one row
    const TileLayout L = tile_layout(p.M, klen, p.rows_per_cta, sb);
    const uint32_t tile = smem_u32(smem_raw);
    uint8_t* img = smem_raw + L.img;
    float* res = reinterpret_cast<float*>(smem_raw + L.res);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + L.bars);
    Shared sh;
    sh.qa_row = (uint32_t)qa_row_stride(klen);
    sh.qa = smem_u32(img);
    sh.ds = sh.qa + (uint32_t)p.M * sh.qa_row;
    sh.stage = tile;

    // 1. every row slice requested at once, before the dependency wait (the
    // lanes of warp 0 share the issuing; one barrier per group of P rows)
    if (warp == 0) {
        if (lane == 0) {
            for (int gi = 0; gi < ngroups; ++gi) mbar_init(&bars[gi], 1);
            fence_mbar_init();
        }
        __syncwarp();
        for (int gi = lane; gi < ngroups; gi += 32) {
            const int r = gi * P, nr = min(P, rows - r);
            mbar_arrive_expect_tx(&bars[gi], (uint32_t)nr * sb);
            for (int j = 0; j < nr; ++j)
                bulk_g2s_u32(tile + (uint32_t)(r + j) * sb, p.w + (row0 + r + j) * p.rb + (int64_t)kb0 * bb, sb,
                             &bars[gi]);
        }
    }
    pdl_launch_dependents();

    // 2. the producer of X has finished: the tile's residual values are read
    // now (one round trip for all of them, under the quantizer) and this K
    // slice is quantized
    pdl_wait();
    const bool res_now = p.residual != nullptr;
    float res0 = 0.f;   // this thread's first residual value, held until after the quantizer
    if (res_now && tid < p.M * rows) {
        const int m = tid / rows, r = tid - m * rows;
        res0 = load_act(p.residual, p.ydt, (int64_t)m * p.N + row0 + r);
    }
    {
        const int rounds = (4 * p.M * (klen / 32) + NT - 1) / NT;   // quarters per thread
        if (rounds >= 4) quantize_slice<4>(p, 0, klen, img, tid, NT);
        else if (rounds >= 2) quantize_slice<2>(p, 0, klen, img, tid, NT);
        else quantize_slice<1>(p, 0, klen, img, tid, NT);
    }
    if (res_now) {
        if (tid < p.M * rows) res[(tid / rows) * p.rows_per_cta + tid % rows] = res0;
        for (int i = tid + NT; i < p.M * rows; i += NT) {
            const int m = i / rows, r = i - m * rows;
            res[m * p.rows_per_cta + r] = load_act(p.residual, p.ydt, (int64_t)m * p.N + row0 + r);
        }
    }
    __syncthreads();   // the image, and the barrier initialisation, are visible
    if (DUMP && row0 == 0) {
        for (int i = tid; i < p.M * klen; i += NT) {
            const int m = i / klen, k = i % klen;
            const uint32_t a = sh.qa + (uint32_t)m * sh.qa_row + qa_pos((uint32_t)k);
            if (p.dbg_qa) p.dbg_qa[(int64_t)m * p.K + k] = (int8_t)(lds32(a & ~3u) >> (8 * (a & 3)));
        }
        for (int i = tid; i < p.M * nbs; i += NT) {
            const int m = i / nbs, b = i % nbs;
            const uint4 e = lds128(sh.ds + 16u * i);
            const int64_t o = (int64_t)m * (p.K / 32) + b;
            if (p.dbg_da) p.dbg_da[o] = __uint_as_float(e.x);
            if (p.dbg_s) p.dbg_s[o] = (int32_t)(e.z + e.w);
        }
    }

    // 3. rows: lane -> (row of the pass, unit); a segmented shuffle reduction
    using Act = ActSlice<MT, AREG, 8, 4>;
    const int seg = U < 32 ? U : 32;
    const int sub_row = U < 32 ? lane / U : 0;
    const int u0 = U < 32 ? lane % U : lane;
    const bool lane_on = U >= 32 || lane < P * U;
    const int seg_end = (lane / seg) * seg + seg;
    const bool head = lane_on && (lane % seg) == 0;
    Act fixed;
    if (U <= 32) fixed.init(sh, 128 * u0, nbs);
    for (int g0 = warp; g0 < ngroups; g0 += TR * NW) {
        // TR row groups per iteration: g0, g0 + NW, ...
        int rr[TR];
        bool vv[TR];
        int64_t nn[TR];
        float acc[TR][MT];
#pragma unroll
        for (int t = 0; t < TR; ++t) {
            const int gi = g0 + t * NW;
            if (gi < ngroups) mbar_wait(&bars[gi], 0, p.status);
            rr[t] = gi * P + sub_row;
            vv[t] = lane_on && gi < ngroups && rr[t] < rows;
            nn[t] = row0 + rr[t];
#pragma unroll
            for (int m = 0; m < MT; ++m) acc[t][m] = 0.f;
        }
        if (U <= 32) {
            FragQ45<QT> f[TR];
            const FragQ45<QT>* fr[TR];
#pragma unroll
            for (int t = 0; t < TR; ++t) {
                if (vv[t]) f[t].load(tile + (uint32_t)rr[t] * sb + (uint32_t)(u0 >> 1) * bb, u0 & 1);
                fr[t] = &f[t];
            }
            bool any = false;
#pragma unroll
            for (int t = 0; t < TR; ++t) any |= vv[t];
            if (any) unit_q45k<QT, MT, TR, Act, DUMP>(p, fr, fixed, kb0 + (u0 >> 1), u0 & 1, acc, nn, vv);
        } else {
#pragma unroll
            for (int t = 0; t < TR; ++t) {
                if (!vv[t]) continue;
                for (int u = u0; u < U; u += 32) {
                    FragQ45<QT> f;
                    f.load(tile + (uint32_t)rr[t] * sb + (uint32_t)(u >> 1) * bb, u & 1);
                    ActSlice<MT, false, 8, 4> a;
                    a.init(sh, 128 * u, nbs);
                    const FragQ45<QT>* fr[1] = {&f};
                    float(*a1)[MT] = reinterpret_cast<float(*)[MT]>(&acc[t][0]);
                    unit_q45k<QT, MT, 1, ActSlice<MT, false, 8, 4>, DUMP>(p, fr, a, kb0 + (u >> 1), u & 1, a1,
                                                                        &nn[t], &vv[t]);
                }
            }
        }
#pragma unroll
        for (int t = 0; t < TR; ++t) {
            if (seg == 32) {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc[t][m] += __shfl_xor_sync(0xffffffffu, acc[t][m], o);
                }
            } else {
#pragma unroll
                for (int m = 0; m < MT; ++m) {
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) {
                        const float tt = __shfl_down_sync(0xffffffffu, acc[t][m], o);
                        if (lane + o < seg_end) acc[t][m] += tt;
                    }
                }
            }
            if (head && vv[t]) {
                for (int m = 0; m < p.M && m < MT; ++m) {
                    float v = acc[t][m];
                    if (p.residual) v += res[m * p.rows_per_cta + rr[t]];
                    store_out(p.y, p.ydt, (int64_t)m * p.N + nn[t], v);
                }
            }
        }
    }

}

// ------------------------------------------------------------------ pair kernel (M = 2..8)
// Q4_K / Q5_K blocks, 2 <= M <= 8, K a multiple of 2048, when a CTA's rows of W
// and the activation image fit in half of an SM's shared memory.  Rows are
// staged whole, as in the tile kernel (two CTAs per SM, the next call's weights
// stream under this call's compute); the image comes from the quantizer kernel.
// A lane owns one 64-value "pair" of K -- the two 32-value sub-blocks whose
// codes share the same 32 qs bytes (low / high nibbles) -- for every row of the
// CTA, so its activation codes and block scales for all M rows are loaded into
// registers once; a warp covers 2048 values of a row, K/2048 warps span a row,
// and their partial sums meet in shared memory.  The M sums of a row are
// reduced across the warp with a transposed butterfly (each step halves the
// values a lane keeps), far fewer shuffles than M separate reductions.
constexpr int kPairWarps = 8;

struct PairLayout {
    int64_t img, res, part, bars, total;
};
__host__ __device__ inline PairLayout pair_layout(int64_t M, int64_t K, int64_t rows_per_cta, int64_t rb) {
    PairLayout L;
    const int64_t KQ = K / 2048;
    L.img = ceil_div(rows_per_cta * rb, 128) * 128;
    L.res = L.img + ceil_div(act_image_bytes(M, K), 16) * 16;
    L.part = L.res + ceil_div(4 * M * rows_per_cta, 16) * 16;
    L.bars = L.part + ceil_div(4 * M * rows_per_cta * KQ, 16) * 16;
    L.total = L.bars + 8 * (rows_per_cta + 1);
    return L;
}

// Transposed butterfly over the 32 lanes: on return, lane l (with l % (32/MT)
// == 0) holds the warp total of value m = l / (32/MT) in v[0].
template <int MT>
__device__ __forceinline__ void warp_sum_transposed(float (&v)[MT], int lane) {
    int n = MT;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        if (n > 1) {
            const bool upper = (lane & o) != 0;
            const int h = n >> 1;
#pragma unroll
            for (int i = 0; i < MT / 2; ++i) {
                if (i < h) {
                    const float keep = upper ? v[h + i] : v[i];
                    const float send = upper ? v[i] : v[h + i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            n = h;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
}

template <int QT, int MT, bool DUMP>
__global__ void __launch_bounds__(kPairWarps * 32, 2) gemv_pair_kernel(const GemvParams p) {
    constexpr int NW = kPairWarps, NT = NW * 32;
    constexpr int bb = QT == GGUF_Q4_K ? 144 : 176;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nb = (int)(p.K / 32);
    const int64_t row0 = (int64_t)blockIdx.x * p.rows_per_cta;
    const int rows = (int)min(p.rows_per_cta, p.N - row0);
    const int KQ = (int)(p.K / 2048), RG = NW / KQ;   // warps per row, row groups
    const int kq = warp % KQ, rg = warp / KQ;
    const uint32_t rb = (uint32_t)p.rb;
    const PairLayout L = pair_layout(p.M, p.K, p.rows_per_cta, p.rb);
    const uint32_t tile = smem_u32(smem_raw);
    uint8_t* img = smem_raw + L.img;
    float* res = reinterpret_cast<float*>(smem_raw + L.res);
    float* part = reinterpret_cast<float*>(smem_raw + L.part);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem_raw + L.bars);   // [rows_per_cta] rows, then the image
    const uint32_t qa_row = (uint32_t)qa_row_stride(p.K);
    const uint32_t qa = smem_u32(img), ds = qa + (uint32_t)p.M * qa_row;

    // 1. every row requested at once, before the dependency wait
    if (warp == 0) {
        if (lane == 0) {
            for (int r = 0; r <= (int)p.rows_per_cta; ++r) mbar_init(&bars[r], 1);
            fence_mbar_init();
        }
        __syncwarp();
        for (int r = lane; r < rows; r += 32) {
            mbar_arrive_expect_tx(&bars[r], rb);
            bulk_g2s_u32(tile + (uint32_t)r * rb, p.w + (row0 + r) * p.rb, rb, &bars[r]);
        }
    }
    __syncthreads();   // every barrier is initialised before any thread waits on one
    pdl_launch_dependents();

    // 2. after the producer of X: the quantized image (one bulk copy) and the
    // tile's residual values
    pdl_wait();
    uint64_t* img_bar = &bars[p.rows_per_cta];
    if (tid == 0) {
        const uint32_t bytes = (uint32_t)act_image_bytes(p.M, p.K);
        mbar_arrive_expect_tx(img_bar, bytes);
        bulk_g2s_u32(qa, p.act_image, bytes, img_bar);
    }
    float res0 = 0.f;
    if (p.residual && tid < p.M * rows)
        res0 = load_act(p.residual, p.ydt, (int64_t)(tid / rows) * p.N + row0 + tid % rows);
    mbar_wait(img_bar, 0, p.status);
    if (p.residual) {
        if (tid < p.M * rows) res[(tid / rows) * p.rows_per_cta + tid % rows] = res0;
        for (int i = tid + NT; i < p.M * rows; i += NT)
            res[(i / rows) * p.rows_per_cta + i % rows] =
                load_act(p.residual, p.ydt, (int64_t)(i / rows) * p.N + row0 + i % rows);
    }
    __syncthreads();
    if (DUMP && blockIdx.x == 0) {
        for (int64_t i = tid; i < (int64_t)p.M * p.K; i += NT) {
            const uint32_t a = qa + (uint32_t)(i / p.K) * qa_row + qa_pos((uint32_t)(i % p.K));
            if (p.dbg_qa) p.dbg_qa[i] = (int8_t)(lds32(a & ~3u) >> (8 * (a & 3)));
        }
        for (int i = tid; i < p.M * nb; i += NT) {
            const uint4 e = lds128(ds + 16u * i);
            if (p.dbg_da) p.dbg_da[i] = __uint_as_float(e.x);
            if (p.dbg_s) p.dbg_s[i] = (int32_t)(e.z + e.w);
        }
    }

    // 3. this lane's pair: values 64*pi .. 64*pi + 63 of K, i.e. sub-blocks
    // jlo = 2*pp (low nibbles) and jlo + 1 (high nibbles) of super-block kb
    const int pi = kq * 32 + lane;
    const int kb = pi >> 2, pp = pi & 3, jlo = 2 * pp;
    uint32_t code[MT][16];
    float da_lo[MT], da_hi[MT], das_lo[MT], das_hi[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
        if (m < p.M) {
            const uint32_t a = qa + (uint32_t)m * qa_row + qa_pos((uint32_t)(64 * pi));
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint4 w4 = lds128(a + 16 * c);
                code[m][4 * c] = w4.x; code[m][4 * c + 1] = w4.y; code[m][4 * c + 2] = w4.z; code[m][4 * c + 3] = w4.w;
            }
            const uint4 e0 = lds128(ds + 16u * (uint32_t)(m * nb + 2 * pi));
            const uint4 e1 = lds128(ds + 16u * (uint32_t)(m * nb + 2 * pi + 1));
            da_lo[m] = __uint_as_float(e0.x); das_lo[m] = __uint_as_float(e0.y);
            da_hi[m] = __uint_as_float(e1.x); das_hi[m] = __uint_as_float(e1.y);
        } else {
#pragma unroll
            for (int c = 0; c < 16; ++c) code[m][c] = 0u;
            da_lo[m] = da_hi[m] = das_lo[m] = das_hi[m] = 0.f;
        }
    }
    const uint32_t rot_lo = (uint32_t)(4 - jlo) & 31u, rot_hi = (uint32_t)(3 - jlo) & 31u;
    const uint32_t blk_off = (uint32_t)kb * bb;

    // 4. rows of this warp's row group
    for (int r = rg; r < rows; r += RG) {
        mbar_wait(&bars[r], 0, p.status);
        const uint32_t blk = tile + (uint32_t)r * rb + blk_off;
        const uint4 hdr = lds128(blk);
        const float d = f16_bits_to_float(hdr.x), dmin = f16_bits_to_float(hdr.x >> 16);
        // 6-bit scale / min of sub-blocks jlo and jlo + 1 (GGUF packing)
        int sc0, sc1, mn0, mn1;
        {
            const uint32_t s0 = hdr.y, s1 = hdr.z, s2 = hdr.w;   // scale bytes 0-3, 4-7, 8-11
            const uint32_t scw = pp < 2 ? (s0 & 0x3F3F3F3Fu) : ((s2 & 0x0F0F0F0Fu) | ((s0 >> 2) & 0x30303030u));
            const uint32_t mnw = pp < 2 ? (s1 & 0x3F3F3F3Fu) : (((s2 >> 4) & 0x0F0F0F0Fu) | ((s1 >> 2) & 0x30303030u));
            const int b = jlo & 3;
            sc0 = (int)((scw >> (8 * b)) & 0xFF); sc1 = (int)((scw >> (8 * b + 8)) & 0xFF);
            mn0 = (int)((mnw >> (8 * b)) & 0xFF); mn1 = (int)((mnw >> (8 * b + 8)) & 0xFF);
        }
        const uint32_t qs = blk + (QT == GGUF_Q5_K ? 48u : 16u) + 32u * (uint32_t)pp;
        const uint4 q0 = lds128(qs), q1 = lds128(qs + 16);
        uint4 h0 = make_uint4(0, 0, 0, 0), h1 = h0;
        if constexpr (QT == GGUF_Q5_K) { h0 = lds128(blk + 16); h1 = lds128(blk + 32); }
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t w = comp(i < 4 ? q0 : q1, i);
            lo[i] = w & 0x0F0F0F0Fu;
            hi[i] = (w >> 4) & 0x0F0F0F0Fu;
            if constexpr (QT == GGUF_Q5_K) {
                const uint32_t hb = comp(i < 4 ? h0 : h1, i);
                lo[i] |= __funnelshift_l(hb, hb, rot_lo) & 0x10101010u;
                hi[i] |= __funnelshift_l(hb, hb, rot_hi) & 0x10101010u;
            }
        }
        float acc[MT];
        const float fmn0 = (float)mn0, fmn1 = (float)mn1;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            int Da = 0, Db = 0, Ea = 0, Eb = 0;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                Da = dp4a(lo[i], code[m][i], Da);
                Db = dp4a(lo[4 + i], code[m][4 + i], Db);
                Ea = dp4a(hi[i], code[m][8 + i], Ea);
                Eb = dp4a(hi[4 + i], code[m][12 + i], Eb);
            }
            const int D0 = Da + Db, D1 = Ea + Eb;
            if (DUMP && p.dbg_D && m < p.M) {
                dump_D(p, m, row0 + r, 2 * pi, 32, D0);
                dump_D(p, m, row0 + r, 2 * pi + 1, 32, D1);
            }
            const float sd = da_lo[m] * (float)(sc0 * D0) + da_hi[m] * (float)(sc1 * D1);
            const float sm = das_lo[m] * fmn0 + das_hi[m] * fmn1;
            acc[m] = d * sd - dmin * sm;
        }
        warp_sum_transposed<MT>(acc, lane);
        const int span = 32 / MT;
        if (lane % span == 0) {
            const int m = lane / span;
            if (m < p.M) part[((int64_t)r * KQ + kq) * p.M + m] = acc[0];
        }
    }

    // 5. the K/2048 partials of each row, + residual, stored
    __syncthreads();
    for (int i = tid; i < p.M * rows; i += NT) {
        const int m = i / rows, r = i % rows;
        float v = 0.f;
        for (int q = 0; q < KQ; ++q) v += part[((int64_t)r * KQ + q) * p.M + m];
        if (p.residual) v += res[m * p.rows_per_cta + r];
        store_out(p.y, p.ydt, (int64_t)m * p.N + row0 + r, v);
    }
}

// ------------------------------------------------------------------ row-lane kernel (M = 1..4)
// Q4_K / Q5_K blocks, when a CTA's rows of W (at most 64) and the activation
// image fit in half of an SM's shared memory.  As in the tile kernel, the
// CTA requests all of its rows with bulk copies at launch (two CTAs share an
// SM, so the next call's weights stream in under this call's compute) and,
// after its dependency wait, quantizes the M activation rows itself: one
// kernel and one wait per call for every M up to 4.
// The mapping is transposed with respect to the other kernels: a lane owns a
// weight ROW and a warp owns a set of 128-value units along K (unit u goes to
// warp u % NW).  All lanes of a warp therefore read the same activation codes
// and block entries at the same time (warp-uniform shared-memory addresses,
// served as broadcasts), every row of the CTA is handled in one round instead
// of one row per warp per round, and the rows' bytes sit at a pitch of an odd
// number of 16-byte chunks, so the eight lanes of a quarter-warp reading the
// same field of eight consecutive rows hit eight different bank groups.
// Each warp leaves one partial sum per (row, activation row) in shared
// memory; the last phase adds the warps' partials in warp order, then the
// residual, and stores.
// With CL > 1 the grid runs in clusters of CL CTAs that share the activation
// quantization: each CTA quantizes K / CL of X and stores the codes into all
// CL images (distributed shared memory), which divides the X reads and the
// quantizer's arithmetic of every CTA by CL.  A residual value is loaded right
// after the dependency wait and held in a register until the store, so its
// latency is hidden under the rows phase.
__host__ __device__ constexpr int rowlane_warps(int mt) { return 16; }

// CTAs per cluster of the row-lane kernel: two from M = 2 on, none at M = 1
// (measured on Q5_K 4096 x 4096, chained calls, us at M = 1 / 2 / 4: one CTA
// 4.20 / 5.48 / 8.17, pairs 4.22 / 4.66 / 6.37, fours 5.06 / 6.60 / 9.86).  GGUF_MM_GEMV_CLUSTER (1, 2 or 4) in the environment, read
// at each call, overrides it for comparison runs.
inline int rowlane_cluster(int64_t M) {
    const char* env = std::getenv("GGUF_MM_GEMV_CLUSTER");
    if (env && (env[0] == '1' || env[0] == '2' || env[0] == '4') && env[1] == 0) return env[0] - '0';
    return M >= 2 ? 2 : 1;
}

struct RowLaneLayout {
    int64_t pitch, img, part, res, bar, total;
};
__host__ __device__ inline RowLaneLayout rowlane_layout(int64_t M, int64_t K, int64_t rows_per_cta, int64_t rb,
                                                        int nw) {
    RowLaneLayout L;
    L.pitch = ((rb / 16) % 2 == 0) ? rb + 16 : rb;      // odd number of 16-byte chunks per row
    L.img = ceil_div(rows_per_cta * L.pitch, 128) * 128;
    L.part = L.img + ceil_div(act_image_bytes(M, K), 16) * 16;
    const int64_t mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : 8;   // the kernel's row stride of partials
    L.res = L.part + ceil_div(4 * (int64_t)nw * rows_per_cta * mt, 16) * 16;
    L.bar = L.res + ceil_div(4 * M * rows_per_cta, 16) * 16;
    L.total = L.bar + 16;
    return L;
}

template <int QT, int MT, int RI, bool DUMP, int CL>
__global__ void __launch_bounds__(rowlane_warps(MT) * 32, 2) gemv_rowlane_kernel(const GemvParams p) {
    constexpr int NW = rowlane_warps(MT), NT = NW * 32;
    constexpr int bb = QT == GGUF_Q4_K ? 144 : 176;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row0 = (int64_t)blockIdx.x * p.rows_per_cta;
    // 1 .. 32 * RI (0 for a CTA that only rounds the grid up to whole clusters)
    const int rows = (int)max((int64_t)0, min(p.rows_per_cta, p.N - row0));
    const int rpc = (int)p.rows_per_cta;
    const int nb = (int)(p.K / 32), U = (int)(p.K / 128);
    const RowLaneLayout L = rowlane_layout(p.M, p.K, p.rows_per_cta, p.rb, NW);
    const uint32_t tile = smem_u32(smem_raw);
    const uint32_t pitch = (uint32_t)L.pitch, rb = (uint32_t)p.rb;
    uint8_t* img = smem_raw + L.img;
    float* part = reinterpret_cast<float*>(smem_raw + L.part);   // [NW][rows_per_cta][MT]
    float* res = reinterpret_cast<float*>(smem_raw + L.res);     // [M][rows_per_cta]
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem_raw + L.bar);

    // 1. every row of the CTA requested at once, before the dependency wait;
    // the same barrier counts the other cluster CTAs' parts of the image
    if (warp == 0) {
        if (lane == 0) {
            mbar_init(bar, 1);
            fence_mbar_init();
            mbar_arrive_expect_tx(bar, (uint32_t)rows * rb + (uint32_t)cluster_xbytes(CL, p.M, p.K));
        }
        __syncwarp();
        for (int r = lane; r < rows; r += 32)
            bulk_g2s_u32(tile + (uint32_t)r * pitch, p.w + (row0 + r) * p.rb, rb, bar);
    }
    // this CTA is running and its barrier initialised (waited on before the
    // first store into another CTA)
    if constexpr (CL > 1) cluster_arrive_relaxed();
    pdl_launch_dependents();

    // 2. after the producer of X: the tile's residual values (one load per
    // thread, issued before the quantizer) and the activation image
    pdl_wait();
    const bool has_res = p.residual != nullptr;
    float res0 = 0.f;
    if (has_res && tid < p.M * rows) res0 = load_act(p.residual, p.ydt, (int64_t)(tid / rows) * p.N + row0 + tid % rows);
    if constexpr (CL > 1) {
        cluster_wait_acquire();   // every CTA of the cluster is running: its image may be written
        const int rounds = (4 * p.M * nb / CL + NT - 1) / NT;
        // (one quarter per round for Q5_K at 3-4 rows keeps its rows phase free
        // of register spills: M = 4 in pairs 7.02 -> 6.37 us)
        if (!(QT == GGUF_Q5_K && MT == 4) && rounds >= 2) quantize_cluster<CL, 2>(p, smem_u32(img), smem_u32(bar), tid, NT);
        else quantize_cluster<CL, 1>(p, smem_u32(img), smem_u32(bar), tid, NT);
    } else {
        const int rounds = (4 * p.M * nb + NT - 1) / NT;   // quarters per thread
        if (rounds >= 4) quantize_slice<4>(p, 0, (int)p.K, img, tid, NT);
        else if (rounds >= 2) quantize_slice<2>(p, 0, (int)p.K, img, tid, NT);
        else quantize_slice<1>(p, 0, (int)p.K, img, tid, NT);
    }
    // residual values past the first NT through shared memory (the first NT
    // stay in the registers of the threads that store them)
    if (has_res) {
        for (int i = tid + NT; i < p.M * rows; i += NT)
            res[(i / rows) * rpc + i % rows] = load_act(p.residual, p.ydt, (int64_t)(i / rows) * p.N + row0 + i % rows);
    }
    // this CTA's part of the image, the residual values and the barrier's
    // initialisation are visible (the other CTAs' parts arrive on the barrier)
    __syncthreads();
    Shared sh;
    sh.qa_row = (uint32_t)qa_row_stride(p.K);
    sh.qa = smem_u32(img);
    sh.ds = sh.qa + (uint32_t)p.M * sh.qa_row;
    sh.stage = tile;

    // 3. lane = row (lane, lane + 32, ...), warp = units warp, warp + NW, ...
    float acc[RI][MT];
#pragma unroll
    for (int i = 0; i < RI; ++i)
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[i][m] = 0.f;
    const bool ok = __syncthreads_and(mbar_wait(bar, 0, p.status) ? 1 : 0) != 0;   // W and the whole image
    if (DUMP && ok && blockIdx.x == 0) {
        for (int64_t i = tid; i < (int64_t)p.M * p.K; i += NT) {
            const uint32_t a = sh.qa + (uint32_t)(i / p.K) * sh.qa_row + qa_pos((uint32_t)(i % p.K));
            if (p.dbg_qa) p.dbg_qa[i] = (int8_t)(lds32(a & ~3u) >> (8 * (a & 3)));
        }
        for (int i = tid; i < p.M * nb; i += NT) {
            const uint4 e = lds128(sh.ds + 16u * i);
            if (p.dbg_da) p.dbg_da[i] = __uint_as_float(e.x);
            if (p.dbg_s) p.dbg_s[i] = (int32_t)(e.z + e.w);
        }
    }
    if (ok) {
        const uint32_t ds_row = 16u * (uint32_t)nb;
        for (int u = warp; u < U; u += NW) {
            const uint32_t ub = (uint32_t)(u >> 1) * bb;
            const uint32_t qa_u = sh.qa + qa_pos((uint32_t)(128 * u)), ds_u = sh.ds + 64u * (uint32_t)u;
#pragma unroll
            for (int i = 0; i < RI; ++i) {
                const int r = lane + 32 * i;
                if (r < rows) {
                    const uint32_t blk = tile + (uint32_t)r * pitch + ub;
                    if (u & 1) unit_rl<QT, MT, 1, DUMP>(p, blk, qa_u, sh.qa_row, ds_u, ds_row, u >> 1, acc[i], row0 + r);
                    else unit_rl<QT, MT, 0, DUMP>(p, blk, qa_u, sh.qa_row, ds_u, ds_row, u >> 1, acc[i], row0 + r);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < RI; ++i) {
        const int r = lane + 32 * i;
        if (r < rows) {
#pragma unroll
            for (int m = 0; m < MT; ++m) part[(warp * rpc + r) * MT + m] = acc[i][m];
        }
    }
    __syncthreads();

    // 4. the warps' partial sums of each (row, activation row), in warp order, + residual
    // (all NW loads in flight at once; warps that owned no unit wrote zeros)
    for (int t = tid; t < p.M * rows; t += NT) {
        const int m = t / rows, r = t - m * rows;
        float pw[NW];
#pragma unroll
        for (int w = 0; w < NW; ++w) pw[w] = part[(w * rpc + r) * MT + m];
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) v += pw[w];
        if (has_res) v += t == tid ? res0 : res[m * rpc + r];
        store_out(p.y, p.ydt, (int64_t)m * p.N + row0 + r, v);
    }
}

template <int QT, int MT, int LAYOUT, bool DUMP>
cudaError_t launch_one(const GemvParams& p, int grid, size_t smem, cudaStream_t stream) {
    const int U = (int)(p.K / (block32(QT) ? 32 : 128));
    auto k = gemv_kernel<QT, MT, LAYOUT, false, DUMP>;
    if constexpr (MT == 1) {
        if (U <= 32) k = gemv_kernel<QT, MT, LAYOUT, true, DUMP>;
    }
    int threads = p.direct ? direct_threads(MT) : kThreads;
    int cl = 1;   // CTAs per cluster
    if constexpr (QT == GGUF_Q4_K || QT == GGUF_Q5_K || (QT == GGUF_Q6_K && LAYOUT == GGUF_LAYOUT_Q6K_PLANES)) {
        if (p.direct) k = gemv_direct_kernel<QT, MT, DUMP>;
    }
    if constexpr ((QT == GGUF_Q4_K || QT == GGUF_Q5_K) && LAYOUT == GGUF_LAYOUT_BLOCKS) {
        if constexpr (MT == 1) {
            if (p.tile == 1) {
                k = gemv_tile_kernel<QT, MT, DUMP>;
                threads = tile_warps(MT) * 32;
            }
        }
        if constexpr (MT >= 2 && MT <= 4) {
            if (p.tile == 2) {
                k = gemv_pair_kernel<QT, MT, DUMP>;
                threads = kPairWarps * 32;
            }
        }
        if constexpr (MT <= 4) {
            if (p.tile == 3) {
                k = p.rows_per_cta > 32   ? gemv_rowlane_kernel<QT, MT, 2, DUMP, 1>
                    : p.cluster == 4      ? gemv_rowlane_kernel<QT, MT, 1, DUMP, 4>
                    : p.cluster == 2      ? gemv_rowlane_kernel<QT, MT, 1, DUMP, 2>
                                          : gemv_rowlane_kernel<QT, MT, 1, DUMP, 1>;
                threads = rowlane_warps(MT) * 32;
                cl = p.rows_per_cta > 32 ? 1 : p.cluster;
            }
        }
    }
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)cl;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = cl > 1 ? 2 : 1;
    if (grid % cl != 0) return cudaErrorInvalidConfiguration;
    return cudaLaunchKernelEx(&cfg, k, p);
}

template <int QT, int LAYOUT, bool DUMP>
cudaError_t launch_mt(const GemvParams& p, int grid, size_t smem, cudaStream_t s) {
    if (p.M <= 1) return launch_one<QT, 1, LAYOUT, DUMP>(p, grid, smem, s);
    if (p.M <= 2) return launch_one<QT, 2, LAYOUT, DUMP>(p, grid, smem, s);
    if (p.M <= 4) return launch_one<QT, 4, LAYOUT, DUMP>(p, grid, smem, s);
    return launch_one<QT, 8, LAYOUT, DUMP>(p, grid, smem, s);
}

template <bool DUMP>
cudaError_t launch_dispatch(const GemvParams& p, int grid, size_t smem, cudaStream_t s) {
    switch (p.qtype) {
        case GGUF_Q4_0: return launch_mt<GGUF_Q4_0, GGUF_LAYOUT_BLOCKS, DUMP>(p, grid, smem, s);
        case GGUF_Q4_1: return launch_mt<GGUF_Q4_1, GGUF_LAYOUT_BLOCKS, DUMP>(p, grid, smem, s);
        case GGUF_Q5_0: return launch_mt<GGUF_Q5_0, GGUF_LAYOUT_BLOCKS, DUMP>(p, grid, smem, s);
        case GGUF_Q5_1: return launch_mt<GGUF_Q5_1, GGUF_LAYOUT_BLOCKS, DUMP>(p, grid, smem, s);
        case GGUF_Q8_0: return launch_mt<GGUF_Q8_0, GGUF_LAYOUT_BLOCKS, DUMP>(p, grid, smem, s);
        case GGUF_Q2_K: return launch_mt<GGUF_Q2_K, GGUF_LAYOUT_BLOCKS, DUMP>(p, grid, smem, s);
        case GGUF_Q3_K: return launch_mt<GGUF_Q3_K, GGUF_LAYOUT_BLOCKS, DUMP>(p, grid, smem, s);
        case GGUF_Q4_K: return launch_mt<GGUF_Q4_K, GGUF_LAYOUT_BLOCKS, DUMP>(p, grid, smem, s);
        case GGUF_Q5_K: return launch_mt<GGUF_Q5_K, GGUF_LAYOUT_BLOCKS, DUMP>(p, grid, smem, s);
        case GGUF_Q6_K:
            return p.layout == GGUF_LAYOUT_Q6K_PLANES
                       ? launch_mt<GGUF_Q6_K, GGUF_LAYOUT_Q6K_PLANES, DUMP>(p, grid, smem, s)
                       : launch_mt<GGUF_Q6_K, GGUF_LAYOUT_BLOCKS, DUMP>(p, grid, smem, s);
    }
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ MoE decode form (mul_mv_id)
// A few routed rows (decode: one token, top_k experts): each row is its own
// GEMV against its expert's blocks, so the rows skip routing and grouping and
// go straight through the int8 path -- each CTA takes kMvRows weight rows of
// one routed row's expert and requests its first fragments before it needs
// the activation row.  With at most kMvFuseRows routed rows (QUANT) the CTA
// quantizes its activation row into shared memory itself while they arrive
// (one kernel per call); with more, the rows are quantized once by the
// quantizer kernel and each CTA copies its row's image (the in-CTA quantizer
// repeated by every CTA of a row costs more than the second kernel: 44 vs 36
// us at 128 rows; 5.5 vs 6.5 us at 8).
constexpr int kMvThreads = 256, kMvRows = 32, kMvFuseRows = 8;

template <int QT, bool QUANT, bool DUMP>
__global__ void __launch_bounds__(kMvThreads) moe_mv_kernel(const MoeMvParams mp) {
    constexpr int bb = QT == GGUF_Q4_K ? 144 : 176;
    constexpr int NW = kMvThreads / 32;
    const int p = (int)blockIdx.y;                      // routed row: token * top_k + slot
    const int e = mp.ids[p];
    if (e < 0 || e >= mp.n_expert) return;              // no expert: the row is left untouched
    const int64_t arow = mp.per_slot ? p : p / mp.top_k;   // its activation row
    const int64_t row0 = (int64_t)blockIdx.x * kMvRows;
    const int64_t row_end = min(mp.N, row0 + kMvRows);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = (int)(mp.K / 32);
    const uint32_t qa_row = (uint32_t)qa_row_stride(mp.K);
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int U = (int)(mp.K / 128);                    // units per row
    const int seg = U < 32 ? U : 32;
    const int P = U < 32 ? 32 / U : 1;                  // rows per warp pass
    const int u0 = U < 32 ? lane % U : lane;
    const int sub_row = U < 32 ? lane / U : 0;
    const bool lane_on = U >= 32 || lane < P * U;
    const int groups = (int)ceil_div(row_end - row0, P);
    const uint8_t* we = mp.w + (int64_t)e * mp.N * mp.rb;
    auto row_of = [&](int g) { return row0 + (int64_t)g * P + sub_row; };
    auto fetch = [&](FragQ45<QT>& f, int g, int u) {
        if (g < groups && lane_on && row_of(g) < row_end)
            load_global<QT>(f, we + row_of(g) * mp.rb + (int64_t)(u >> 1) * bb, u & 1);
    };
    if constexpr (!QUANT) {
        // this row's image (codes [qa_row] then entries [nb]) from the workspace
        const uint4* sc = reinterpret_cast<const uint4*>(mp.image + arow * qa_row);
        const uint4* se = reinterpret_cast<const uint4*>(mp.image + mp.rows * (int64_t)qa_row + arow * nb * 16);
        uint4* dc = reinterpret_cast<uint4*>(smem_raw);
        uint4* de = reinterpret_cast<uint4*>(smem_raw + qa_row);
        for (int i = threadIdx.x; i < (int)(qa_row / 16); i += kMvThreads) dc[i] = sc[i];
        for (int i = threadIdx.x; i < nb; i += kMvThreads) de[i] = se[i];
    }
    // one unit per lane and row (K <= 4096): this warp's first two row groups
    // are requested together, before the activation row has landed
    FragQ45<QT> f0, f1;
    if (U <= 32) {
        fetch(f0, warp, u0);
        fetch(f1, warp + NW, u0);
    }
    if constexpr (QUANT) {
        // the activation row -> codes [qa_row] then entries [nb] in shared memory
        GemvParams q{};
        q.x = static_cast<const uint8_t*>(mp.x) + arow * mp.K * (mp.xdt == GGUF_DT_F32 ? 4 : 2);
        q.xdt = mp.xdt;
        q.M = 1;
        q.K = mp.K;
        const int rounds = (4 * nb + kMvThreads - 1) / kMvThreads;   // quarters per thread
        if (rounds >= 4) quantize_slice<4>(q, 0, (int)mp.K, smem_raw, threadIdx.x, kMvThreads);
        else if (rounds >= 2) quantize_slice<2>(q, 0, (int)mp.K, smem_raw, threadIdx.x, kMvThreads);
        else quantize_slice<1>(q, 0, (int)mp.K, smem_raw, threadIdx.x, kMvThreads);
    }
    __syncthreads();
    Shared sh;
    sh.qa = smem_u32(smem_raw);
    sh.qa_row = qa_row;
    sh.ds = sh.qa + qa_row;
    sh.stage = 0;
    GemvParams gp{};
    gp.M = 1;
    gp.K = mp.K;
    gp.N = mp.N;
    if constexpr (DUMP) {
        if (blockIdx.x == 0) {
            for (int64_t k = threadIdx.x; k < mp.K; k += kMvThreads) {
                const uint32_t a = sh.qa + qa_pos((uint32_t)k);
                if (mp.dbg_qa) mp.dbg_qa[(int64_t)p * mp.K + k] = (int8_t)(lds32(a & ~3u) >> (8 * (a & 3)));
            }
            for (int b = threadIdx.x; b < nb; b += kMvThreads) {
                const uint4 en = lds128(sh.ds + 16u * b);
                if (mp.dbg_da) mp.dbg_da[(int64_t)p * nb + b] = __uint_as_float(en.x);
                if (mp.dbg_s) mp.dbg_s[(int64_t)p * nb + b] = (int32_t)(en.z + en.w);
            }
        }
        gp.dbg_D = mp.dbg_D ? mp.dbg_D + (int64_t)p * mp.N * nb : nullptr;   // [N][K/32] of row p
    }
    const int seg_end = (lane / seg) * seg + seg;
    const bool head = lane_on && (lane % seg) == 0;
    using Act = ActSlice<1, false, 8, 4>;
    auto compute = [&](const FragQ45<QT>& f, int g, int u, float (&acc)[1][1]) {
        if (!(g < groups && lane_on && row_of(g) < row_end)) return;
        Act a;
        a.init(sh, 128 * u, nb);
        const FragQ45<QT>* fr[1] = {&f};
        const int64_t nn[1] = {row_of(g)};
        const bool on[1] = {true};
        unit_q45k<QT, 1, 1, Act, DUMP>(gp, fr, a, u >> 1, u & 1, acc, nn, on);
    };
    auto finish = [&](float (&acc)[1][1], int g) {
        if (seg == 32) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[0][0] += __shfl_xor_sync(0xffffffffu, acc[0][0], o);
        } else {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float t = __shfl_down_sync(0xffffffffu, acc[0][0], o);
                if (lane + o < seg_end) acc[0][0] += t;
            }
        }
        const int64_t n = row_of(g);
        if (head && g < groups && n < row_end) {
            const int64_t o = (int64_t)p * mp.N + n;
            float v = acc[0][0];
            if (mp.residual) v += load_act(mp.residual, mp.ydt, o);
            store_out(mp.y, mp.ydt, o, v);
        }
    };
    if (U <= 32) {
        for (int g = warp; g < groups; g += 2 * NW) {
            float acc[1][1] = {{0.f}};
            compute(f0, g, u0, acc);
            fetch(f0, g + 2 * NW, u0);
            finish(acc, g);
            acc[0][0] = 0.f;
            compute(f1, g + NW, u0, acc);
            fetch(f1, g + 3 * NW, u0);
            finish(acc, g + NW);
        }
    } else {
        for (int g = warp; g < groups; g += NW) {
            float acc[1][1] = {{0.f}};
            for (int u = u0; u < U; u += 32) {
                fetch(f0, g, u);
                compute(f0, g, u, acc);
            }
            finish(acc, g);
        }
    }
}

}  // namespace

int gemv_plan(GemvParams& p, int num_sms, int max_smem, int* grid, size_t* smem) {
    const int bv = block_values(p.qtype);
    const int bb = block_bytes(p.qtype);
    p.rb = p.K / bv * bb;
    const int64_t act = act_image_bytes(p.M, p.K);
    const int U = (int)(p.K / (block32(p.qtype) ? 32 : 128));
    const int64_t P = U < 32 ? 32 / U : 1;
    const int NW = kThreads / 32;
    // a slot holds one row group plus 16-byte alignment slack (the D plane
    // piece of the planes layout gets its own slack)
    p.stage_bytes = ceil_div(P * p.rb + 48, 16) * 16;
    // one CTA per SM; it keeps to half of the shared memory so that a CTA of
    // the next call on the stream (programmatic dependent launch) fits beside it
    const int64_t half = std::min<int64_t>(max_smem, 232448 / 2 - 1024);
    // one activation row: the tile kernel, when a CTA's rows of W and its image
    // fit beside a second CTA (the quantizer runs inside it; from two rows on the
    // stand-alone quantizer kernel, whose work is not repeated by every CTA, wins)
    p.tile = 0;
    const bool q45 = (p.qtype == GGUF_Q4_K || p.qtype == GGUF_Q5_K) && p.layout == GGUF_LAYOUT_BLOCKS;
    // up to four rows: the row-lane kernel, when a CTA's rows (at most 64, and
    // enough of them to occupy most lanes) and the image fit beside a second CTA
    if (q45 && p.M <= 4 && (p.force < 0 || p.force == GEMV_ROWLANE)) {
        const int64_t rpc_t = ceil_div(p.N, (int64_t)num_sms);
        const int mt = p.M <= 1 ? 1 : p.M <= 2 ? 2 : 4;
        const RowLaneLayout L = rowlane_layout(p.M, p.K, rpc_t, p.rb, rowlane_warps(mt));
        // clusters sharing the quantization (at most 32 rows per CTA): whole
        // clusters, a CTA past N only quantizes
        const int cl = rpc_t <= 32 ? rowlane_cluster(p.M) : 1;
        // one barrier phase counts the CTA's rows and the image parts of the
        // other CTAs (transaction counts stay below 2^20 bytes)
        if (rpc_t <= 64 && (rpc_t >= 16 || p.force == GEMV_ROWLANE) && L.total <= half &&
            rpc_t * p.rb + cluster_xbytes(cl, p.M, p.K) < (int64_t(1) << 20)) {
            p.tile = 3;
            p.direct = 0;
            p.rows_per_cta = rpc_t;
            p.cluster = cl;
            *grid = (int)(ceil_div(ceil_div(p.N, rpc_t), (int64_t)cl) * cl);
            *smem = (size_t)L.total;
            return GGUF_OK;
        }
    }
    if (p.force == GEMV_ROWLANE) return GGUF_ERR_UNSUPPORTED;
    if (q45 && p.M == 1 && (p.force < 0 || p.force == GEMV_TILE)) {
        const int64_t rpc_t = ceil_div(p.N, (int64_t)num_sms);
        const TileLayout L = tile_layout(p.M, p.K, rpc_t, p.rb);
        if (L.total <= half) {
            p.tile = 1;
            p.direct = 0;
            p.rows_per_cta = rpc_t;
            p.stage_bytes = L.img;
            *grid = (int)ceil_div(p.N, rpc_t);
            *smem = (size_t)L.total;
            return GGUF_OK;
        }
    }
    const int64_t rpc = ceil_div(p.N, (int64_t)num_sms);
    // the pair kernel for 2..4 rows: whole rows staged, codes in registers
    if (p.force == GEMV_TILE) return GGUF_ERR_UNSUPPORTED;
    if (q45 && p.M >= 2 && p.M <= 4 && p.K % 2048 == 0 && kPairWarps % (p.K / 2048) == 0 &&
        (p.force < 0 || p.force == GEMV_PAIR)) {
        const PairLayout L = pair_layout(p.M, p.K, rpc, p.rb);
        if (L.total <= half) {
            p.tile = 2;
            p.direct = 0;
            p.rows_per_cta = rpc;
            *grid = (int)ceil_div(p.N, rpc);
            *smem = (size_t)L.total;
            return GGUF_OK;
        }
    }
    if (p.force == GEMV_PAIR) return GGUF_ERR_UNSUPPORTED;
    const int64_t groups_per_warp = ceil_div(ceil_div(rpc, P), NW);
    int64_t R = std::min<int64_t>({groups_per_warp, 8, (half - act) / (NW * p.stage_bytes)});
    if (R < 1) R = std::min<int64_t>({groups_per_warp, 8, (max_smem - act) / (NW * p.stage_bytes)});
    if (R < 1) return GGUF_ERR_UNSUPPORTED;
    p.stages = (int)R;
    p.direct = (p.qtype == GGUF_Q4_K || p.qtype == GGUF_Q5_K ||
                (p.qtype == GGUF_Q6_K && p.layout == GGUF_LAYOUT_Q6K_PLANES)) ? 1 : 0;
    if (p.force == GEMV_STAGED) p.direct = 0;
    if (p.force == GEMV_DIRECT && !p.direct) return GGUF_ERR_UNSUPPORTED;
    p.rows_per_cta = rpc;
    p.chunk_rows = 0;
    *grid = (int)ceil_div(p.N, rpc);
    // + the image barrier (8 bytes, after the per-warp ring barriers)
    // direct: image, its barrier (16 bytes with padding), the residual values
    *smem = p.direct ? (size_t)(act + 16 + 4 * p.M * rpc)
                     : (size_t)(act + NW * R * p.stage_bytes + NW * R * 8 + 8);
    return GGUF_OK;
}

int gemv_kind(const GemvParams& p) {
    return p.tile == 1 ? GEMV_TILE : p.tile == 2 ? GEMV_PAIR : p.tile == 3 ? GEMV_ROWLANE
                                                                           : p.direct ? GEMV_DIRECT : GEMV_STAGED;
}

cudaError_t gemv_launch(const GemvParams& p, int grid, size_t smem, bool dump, cudaStream_t stream) {
    if (p.tile == 1 || p.tile == 3) return dump ? launch_dispatch<true>(p, grid, smem, stream) : launch_dispatch<false>(p, grid, smem, stream);
    // 1. per-32 activation quantizer -> image in the workspace
    const int quarters = 4 * p.M * (int)(p.K / 32);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ceil_div(quarters, 256));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, act_quant_kernel, p);
    if (e != cudaSuccess) return e;
    // 2. the GEMV
    return dump ? launch_dispatch<true>(p, grid, smem, stream) : launch_dispatch<false>(p, grid, smem, stream);
}

size_t gemv_workspace_bytes(int64_t M, int64_t K) { return (size_t)(ceil_div(act_image_bytes(M, K), 256) * 256); }

// ------------------------------------------------------------------ MoE decode form entry
size_t moe_mv_image_bytes(int64_t rows, int64_t K) { return (size_t)(ceil_div(act_image_bytes(rows, K), 256) * 256); }

cudaError_t moe_mv_launch(const MoeMvParams& mp, cudaStream_t stream, bool dump) {
    cudaError_t e = cudaSuccess;
    const bool quant = mp.entries <= kMvFuseRows;
    if (!quant) {
        // the activation rows quantized once, into the workspace image
        GemvParams q{};
        q.x = mp.x;
        q.xdt = mp.xdt;
        q.M = (int)mp.rows;
        q.K = mp.K;
        q.act_image = const_cast<uint8_t*>(mp.image);
        q.status = mp.status;
        const int quarters = 4 * q.M * (int)(mp.K / 32);
        act_quant_kernel<<<(unsigned)ceil_div(quarters, 256), 256, 0, stream>>>(q);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // one CTA per (kMvRows weight rows, routed row); the activation row's image in shared memory
    const size_t smem = (size_t)(qa_row_stride(mp.K) + (mp.K / 32) * 16);
    auto k = mp.qtype == GGUF_Q4_K ? (quant ? moe_mv_kernel<GGUF_Q4_K, true, false> : moe_mv_kernel<GGUF_Q4_K, false, false>)
                                   : (quant ? moe_mv_kernel<GGUF_Q5_K, true, false> : moe_mv_kernel<GGUF_Q5_K, false, false>);
    if (dump)
        k = mp.qtype == GGUF_Q4_K ? (quant ? moe_mv_kernel<GGUF_Q4_K, true, true> : moe_mv_kernel<GGUF_Q4_K, false, true>)
                                  : (quant ? moe_mv_kernel<GGUF_Q5_K, true, true> : moe_mv_kernel<GGUF_Q5_K, false, true>);
    if (smem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
    dim3 grid((unsigned)ceil_div(mp.N, kMvRows), (unsigned)mp.entries);
    k<<<grid, kMvThreads, smem, stream>>>(mp);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ MoE decode form, other formats
// The routed rows' activations quantized once into the workspace image, then
// the staged GEMV kernel in routed mode: grid (row CTAs, routed rows), each
// CTA streaming its rows of the routed row's expert.
template <int QT>
cudaError_t launch_routed(const GemvParams& p, int grid, int rows, size_t smem, cudaStream_t stream) {
    const int U = (int)(p.K / (block32(QT) ? 32 : 128));
    auto k = U <= 32 ? gemv_kernel<QT, 1, GGUF_LAYOUT_BLOCKS, true, false, true>
                     : gemv_kernel<QT, 1, GGUF_LAYOUT_BLOCKS, false, false, true>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, (unsigned)rows);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = p.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, p);
}

int moe_mv_staged_run(const MoeMvParams& mp, int num_sms, int max_smem, cudaStream_t stream) {
    GemvParams q{};
    q.x = mp.x;
    q.xdt = mp.xdt;
    q.M = (int)mp.rows;
    q.K = mp.K;
    q.act_image = const_cast<uint8_t*>(mp.image);
    q.status = mp.status;
    GemvParams p{};
    p.w = mp.w;
    p.qtype = mp.qtype;
    p.layout = GGUF_LAYOUT_BLOCKS;
    p.N = mp.N;
    p.K = mp.K;
    p.x = mp.x;
    p.xdt = mp.xdt;
    p.M = 1;
    p.residual = mp.residual;
    p.y = mp.y;
    p.ydt = mp.ydt;
    p.status = mp.status;
    p.pdl = mp.pdl;
    p.act_image = q.act_image;
    p.force = GEMV_STAGED;
    int grid = 0;
    size_t smem = 0;
    // CTAs sized over the whole batch: two per SM up to 16 routed rows, four
    // above (measured best on 128 experts of 768 x 2048); the plain plan would
    // give every routed row all the SMs, thousands of few-row CTAs
    const int fac = mp.entries <= 16 ? 2 : 4;
    const int per_row = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms, ceil_div((int64_t)fac * num_sms, mp.entries)));
    if (gemv_plan(p, per_row, max_smem, &grid, &smem) != GGUF_OK) return GGUF_ERR_UNSUPPORTED;
    p.ids = mp.ids;
    p.n_expert = mp.n_expert;
    p.route_div = mp.per_slot ? 1 : mp.top_k;
    p.img_rows = mp.rows;
    const int quarters = 4 * q.M * (int)(mp.K / 32);
    act_quant_kernel<<<(unsigned)ceil_div(quarters, 256), 256, 0, stream>>>(q);
    if (cudaGetLastError() != cudaSuccess) return GGUF_ERR_CUDA;
    cudaError_t e = cudaErrorInvalidValue;
    switch (mp.qtype) {
        case GGUF_Q4_0: e = launch_routed<GGUF_Q4_0>(p, grid, mp.entries, smem, stream); break;
        case GGUF_Q4_1: e = launch_routed<GGUF_Q4_1>(p, grid, mp.entries, smem, stream); break;
        case GGUF_Q5_0: e = launch_routed<GGUF_Q5_0>(p, grid, mp.entries, smem, stream); break;
        case GGUF_Q5_1: e = launch_routed<GGUF_Q5_1>(p, grid, mp.entries, smem, stream); break;
        case GGUF_Q8_0: e = launch_routed<GGUF_Q8_0>(p, grid, mp.entries, smem, stream); break;
        case GGUF_Q2_K: e = launch_routed<GGUF_Q2_K>(p, grid, mp.entries, smem, stream); break;
        case GGUF_Q3_K: e = launch_routed<GGUF_Q3_K>(p, grid, mp.entries, smem, stream); break;
        case GGUF_Q6_K: e = launch_routed<GGUF_Q6_K>(p, grid, mp.entries, smem, stream); break;
        default: return GGUF_ERR_UNSUPPORTED;
    }
    return e == cudaSuccess ? GGUF_OK : GGUF_ERR_CUDA;
}

}  // namespace gg
