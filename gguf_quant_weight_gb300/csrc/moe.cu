// MoE expert GEMM (mul_mm_id): Y[t, k, :] = X[t, :] . W_{ids[t,k]}^T (+ residual).
//
// llama.cpp PR #28301 "metal : skip the empty half of the mul_mm_id token
// tile", "Overview" and "Additional information": every routed (token, slot)
// row multiplies its expert's weight; experts receive few rows per ubatch
// (rows per expert ~ ubatch * n_used / n_expert, skewed by routing), so most
// token tiles are underfilled, and the padded rows should cost nothing.
//
// GB300 shape of it, three kernels on the caller's stream:
//   1. route  (one CTA): per-expert row counts, a block-wide scan for each
//      expert's group offset and first work item, the work list of
//      (expert, token tile of up to 128 rows), and the grouped row list
//      (entry = token * top_k + slot of each row, grouped by expert);
//   2. gather: the activation row of every grouped entry, converted to f16,
//      packed contiguously so each token tile is one TMA box;
//   3. the fused tensor-core GEMM in grouped mode: one CTA per (128 weight
//      rows, work item), the expert's GGUF blocks decoded in the kernel, and
//      MMAs issued for round_up(rows, 16) token columns only.
// Nothing waits on the host: the counts never leave the device, so the GEMM
// grid is the upper bound on work items and surplus CTAs exit at once.
//
// Decode form (mul_mv_id): with at most moe_mv_max_rows(qtype) routed rows
// (Q4_K 128: measured against the routed path, 23 vs 33 us at 64 rows, 38 vs
// 44 at 128, 66 vs 54 at 256, Q4_K 128 x 768 x 2048; the other formats' limits
// from the same comparison) every row is a GEMV of its own, on the int8 path of
// the decode GEMV (ov39119's path table sends small batches to the GEMV): no
// routing, no grouping, and CTAs over (weight rows, routed row) instead of a
// tile per expert that decodes 128 rows to f16 for one token column. Q4_K and
// Q5_K use a kernel of their own (one CTA per 32 weight rows of a routed row);
// the other formats the staged GEMV kernel in routed mode.
#include <algorithm>
#include <cstdlib>

#include "common.cuh"
#include "formats.cuh"
#include "gemm.cuh"
#include "gemv.cuh"
#include "moe.cuh"

namespace gg {

namespace {

constexpr int kRouteThreads = 1024;
constexpr int kMoeTile = 128;   // token rows per work item (the GEMM's BN)

// GGUF_MM_MOE_MV=0 in the environment (read at each call) keeps every batch
// on the routed path, for comparison runs
bool mv_form(int qtype, int64_t entries) {
    const char* env = std::getenv("GGUF_MM_MOE_MV");
    if (env && env[0] == '0') return false;
    return entries <= moe_mv_max_rows(qtype);
}

struct MoeLayout {
    int* offsets;   // [E + 1]
    int* ntiles;    // [1]
    int4* tiles;    // [max_tiles]
    int* rows;      // [T * top_k]
    float* xscale;  // [T * top_k] power-of-two scale of each gathered f16 row
    uint16_t* xg;   // [T * top_k, K] f16
    int64_t max_tiles;
    size_t bytes;
};

MoeLayout moe_layout(void* base, int64_t E, int64_t K, int64_t T, int64_t top_k) {
    const int64_t entries = T * top_k;
    MoeLayout L{};
    L.max_tiles = std::min(E, entries) + ceil_div(entries, kMoeTile);
    auto r256 = [](int64_t b) { return ceil_div(b, 256) * 256; };
    int64_t off = 0;
    uint8_t* p = static_cast<uint8_t*>(base);
    auto take = [&](int64_t bytes) { uint8_t* q = p ? p + off : nullptr; off += r256(bytes); return q; };
    L.offsets = reinterpret_cast<int*>(take(4 * (E + 1)));
    L.ntiles = reinterpret_cast<int*>(take(4));
    L.tiles = reinterpret_cast<int4*>(take(16 * L.max_tiles));
    L.rows = reinterpret_cast<int*>(take(4 * entries));
    L.xscale = reinterpret_cast<float*>(take(4 * entries));
    L.xg = reinterpret_cast<uint16_t*>(take(2 * entries * K));
    L.bytes = (size_t)off;
    return L;
}

// Exclusive block-wide prefix sums of two values (1024 threads).
__device__ __forceinline__ void block_scan2(int a, int b, int& ea, int& eb, int& ta, int& tb, int* wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int ia = a, ib = b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int xa = __shfl_up_sync(0xffffffffu, ia, o), xb = __shfl_up_sync(0xffffffffu, ib, o);
        if (lane >= o) { ia += xa; ib += xb; }
    }
    if (lane == 31) { wsum[warp] = ia; wsum[32 + warp] = ib; }
    __syncthreads();
    if (warp == 0) {
        int va = wsum[lane], vb = wsum[32 + lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int xa = __shfl_up_sync(0xffffffffu, va, o), xb = __shfl_up_sync(0xffffffffu, vb, o);
            if (lane >= o) { va += xa; vb += xb; }
        }
        wsum[64 + lane] = va;   // inclusive scan of warp totals
        wsum[96 + lane] = vb;
    }
    __syncthreads();
    const int pa = warp ? wsum[64 + warp - 1] : 0, pb = warp ? wsum[96 + warp - 1] : 0;
    ea = pa + ia - a;
    eb = pb + ib - b;
    ta = wsum[64 + 31];
    tb = wsum[96 + 31];
}

__global__ void __launch_bounds__(kRouteThreads) moe_route_kernel(const int32_t* __restrict__ ids, int total, int E,
                                                                  int max_tiles, int* offsets, int* ntiles,
                                                                  int4* tiles, int* rows) {
    pdl_launch_dependents();   // the gather kernel may launch; it waits for these tables
    extern __shared__ int sm[];
    int* cnt = sm;             // [E] rows per expert
    int* cur = sm + E;         // [E] next free position of each group
    int* wsum = sm + 2 * E;    // [128] scan scratch
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += kRouteThreads) cnt[e] = 0;
    __syncthreads();
    for (int i = tid; i < total; i += kRouteThreads) {
        const int e = ids[i];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    // thread tid owns experts [tid*per, tid*per + per)
    const int per = (E + kRouteThreads - 1) / kRouteThreads;
    const int e0 = tid * per, e1 = min(E, e0 + per);
    int my_rows = 0, my_tiles = 0;
    for (int e = e0; e < e1; ++e) {
        my_rows += cnt[e];
        my_tiles += (cnt[e] + kMoeTile - 1) / kMoeTile;
    }
    int row_base, tile_base, all_rows, all_tiles;
    block_scan2(my_rows, my_tiles, row_base, tile_base, all_rows, all_tiles, wsum);
    for (int e = e0; e < e1; ++e) {
        offsets[e] = row_base;
        cur[e] = row_base;
        for (int s = 0; s < cnt[e]; s += kMoeTile) {
            if (tile_base < max_tiles) tiles[tile_base] = make_int4(e, s, min(kMoeTile, cnt[e] - s), 0);
            ++tile_base;
        }
        row_base += cnt[e];
    }
    if (tid == 0) {
        offsets[E] = all_rows;
        *ntiles = min(all_tiles, max_tiles);
    }
    __syncthreads();
    for (int i = tid; i < total; i += kRouteThreads) {
        const int e = ids[i];
        if (e >= 0 && e < E) rows[atomicAdd(&cur[e], 1)] = i;
    }
}

// One warp per grouped row: its activation row -> f16, 8 values per lane
// step, scaled by 2^-s with s = floor(log2(max |x|)) - 14 so that the row's
// largest magnitude lands in [2^14, 2^15) (a bf16 row beyond f16's range
// stays finite; a row below its normal range keeps its bits); 2^s goes to
// xscale[p] for the GEMM's epilogue.  A power of two is exact; a row holding
// inf or NaN is left unscaled.  The row is x[token] (one row per token,
// shared by its slots) or, in the per-slot form, x[token * top_k + slot]
// (row_div = 1).
__device__ __forceinline__ void load8_16(const uint16_t* src, int xdt, float v[8]) {
    const uint4 t = *reinterpret_cast<const uint4*>(src);
    const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (xdt == GGUF_DT_F16) {
            v[2 * j] = f16_bits_to_float(w4[j] & 0xFFFFu);
            v[2 * j + 1] = f16_bits_to_float(w4[j] >> 16);
        } else {
            v[2 * j] = __uint_as_float(w4[j] << 16);
            v[2 * j + 1] = __uint_as_float(w4[j] & 0xFFFF0000u);
        }
    }
}

// A row of up to 32 lanes x 8 chunks of 8 values is loaded once into
// registers, all loads in flight; longer rows take a second pass.
constexpr int kGatherChunks = 8;

__global__ void __launch_bounds__(256) moe_gather_kernel(const void* __restrict__ x, int xdt, int64_t K, int row_div,
                                                         const int* __restrict__ row_count,
                                                         const int* __restrict__ rows, int64_t cap,
                                                         uint16_t* __restrict__ xg, float* __restrict__ xscale) {
    const int lane = threadIdx.x & 31;
    pdl_launch_dependents();   // the grouped GEMM may launch; it waits for the gathered rows
    pdl_wait();                // the routing tables come from the kernel before
    const int64_t p = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (p >= cap || p >= *row_count) return;
    const int64_t t = rows[p] / row_div;
    const uint16_t* src = static_cast<const uint16_t*>(x) + t * K;
    uint16_t* dst = xg + p * K;
    const int64_t nch = K / 8;
    const bool in_regs = nch <= 32 * kGatherChunks;
    float v[kGatherChunks][8];
    float amax = 0.f;
    bool finite = true;
    if (in_regs) {
#pragma unroll
        for (int c = 0; c < kGatherChunks; ++c)
            if (lane + 32 * c < nch) load8_16(src + 8 * (lane + 32 * c), xdt, v[c]);
#pragma unroll
        for (int c = 0; c < kGatherChunks; ++c) {
            if (lane + 32 * c < nch) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    finite = finite && isfinite(v[c][j]);
                    amax = fmaxf(amax, fabsf(v[c][j]));
                }
            }
        }
    } else {
        for (int64_t ch = lane; ch < nch; ch += 32) {
            float u[8];
            load8_16(src + 8 * ch, xdt, u);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                finite = finite && isfinite(u[j]);
                amax = fmaxf(amax, fabsf(u[j]));
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    finite = __all_sync(0xffffffffu, finite);
    float mul = 1.f, back = 1.f;
    if (finite && amax > 0.f) {
        const int s = max(-100, min(100, ilogbf(amax) - 14));
        mul = ldexpf(1.f, -s);
        back = ldexpf(1.f, s);
    }
    auto store8 = [&](int64_t ch, const float (&u)[8]) {
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 h = __floats2half2_rn(u[2 * j] * mul, u[2 * j + 1] * mul);
            o[j] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(dst + 8 * ch) = make_uint4(o[0], o[1], o[2], o[3]);
    };
    if (in_regs) {
#pragma unroll
        for (int c = 0; c < kGatherChunks; ++c)
            if (lane + 32 * c < nch) store8(lane + 32 * c, v[c]);
    } else {
        for (int64_t ch = lane; ch < nch; ch += 32) {
            float u[8];
            load8_16(src + 8 * ch, xdt, u);
            store8(ch, u);
        }
    }
    if (lane == 0) xscale[p] = back;
}

}  // namespace

int moe_route_debug(const int32_t* ids, int64_t entries, int64_t n_expert, int* offsets, int* ntiles, int4* tiles,
                    int64_t max_tiles, int* rows, cudaStream_t stream) {
    const size_t route_smem = (size_t)(2 * n_expert + 128) * sizeof(int);
    if (route_smem > 48 * 1024 &&
        cudaFuncSetAttribute(moe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)route_smem) !=
            cudaSuccess)
        return GGUF_ERR_CUDA;
    moe_route_kernel<<<1, kRouteThreads, route_smem, stream>>>(ids, (int)entries, (int)n_expert, (int)max_tiles,
                                                              offsets, ntiles, tiles, rows);
    return cudaGetLastError() == cudaSuccess ? GGUF_OK : GGUF_ERR_CUDA;
}

int64_t moe_max_tiles(int64_t n_expert, int64_t entries) { return std::min(n_expert, entries) + ceil_div(entries, kMoeTile); }

bool moe_decode_form(int qtype, int64_t entries) { return mv_form(qtype, entries); }

int moe_mv_max_rows(int qtype) {
    switch (qtype) {
        case GGUF_Q4_K: case GGUF_Q5_K: case GGUF_Q2_K: case GGUF_Q3_K: case GGUF_Q6_K: return kMoeMvRows;
        case GGUF_Q8_0: return 16;
        default: return 32;
    }
}

size_t moe_workspace_bytes(int qtype, int64_t n_expert, int64_t N, int64_t K, int64_t T, int64_t top_k) {
    (void)N;
    // enough for either form, so a comparison run may switch between them
    const size_t routed = moe_layout(nullptr, n_expert, K, T, top_k).bytes;
    if (T * top_k <= kMoeMvRows) return std::max(routed, moe_mv_image_bytes(T * top_k, K));
    return routed;
}

int moe_run(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K, const void* x, int xdt,
            int64_t T, const int32_t* ids, int64_t top_k, const void* residual, void* y, int ydt, void* workspace,
            int num_sms, int* status, cudaStream_t stream, bool per_slot, const MoeMvDump* dump, int pdl, int form) {
    if (K % 256 != 0) return GGUF_ERR_UNSUPPORTED;
    const int64_t entries = T * top_k;
    if (entries > INT32_MAX / 2 || n_expert * N > INT32_MAX) return GGUF_ERR_UNSUPPORTED;
    if (form == 1 && entries > kMoeMvRows) return GGUF_ERR_UNSUPPORTED;
    const bool decode = form < 0 ? mv_form(qtype, entries) : form == 1;
    const bool q45 = qtype == GGUF_Q4_K || qtype == GGUF_Q5_K;
    if (dump && !(decode && q45)) return GGUF_ERR_UNSUPPORTED;
    if (decode) {
        MoeMvParams mp{};
        mp.w = static_cast<const uint8_t*>(w_experts);
        mp.qtype = qtype;
        mp.n_expert = n_expert;
        mp.N = N;
        mp.K = K;
        mp.rb = K / 256 * block_bytes(qtype);
        mp.ids = ids;
        mp.entries = (int)entries;
        mp.top_k = (int)top_k;
        mp.per_slot = per_slot ? 1 : 0;
        mp.x = x;
        mp.xdt = xdt;
        mp.image = static_cast<const uint8_t*>(workspace);
        mp.rows = per_slot ? entries : T;
        mp.residual = residual;
        mp.y = y;
        mp.ydt = ydt;
        mp.status = status;
        mp.pdl = pdl;
        // Q4_K / Q5_K: the decode-form kernel with its row-group fragments;
        // the other formats: the staged GEMV kernel in routed mode
        if (!q45) return moe_mv_staged_run(mp, num_sms, 232448, stream);   // the sm_103 opt-in maximum
        if (dump) {
            mp.dbg_qa = dump->qa;
            mp.dbg_da = dump->da;
            mp.dbg_s = dump->s;
            mp.dbg_D = dump->D;
        }
        return moe_mv_launch(mp, stream, dump != nullptr) == cudaSuccess ? GGUF_OK : GGUF_ERR_CUDA;
    }
    const MoeLayout L = moe_layout(workspace, n_expert, K, T, top_k);
    const size_t route_smem = (size_t)(2 * n_expert + 128) * sizeof(int);
    if (route_smem > 48 * 1024 &&
        cudaFuncSetAttribute(moe_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)route_smem) !=
            cudaSuccess)
        return GGUF_ERR_CUDA;
    moe_route_kernel<<<1, kRouteThreads, route_smem, stream>>>(ids, (int)entries, (int)n_expert, (int)L.max_tiles,
                                                              L.offsets, L.ntiles, L.tiles, L.rows);
    if (cudaGetLastError() != cudaSuccess) return GGUF_ERR_CUDA;
    {   // a programmatic dependent of the routing kernel
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)ceil_div(entries, 8));
        cfg.blockDim = dim3(256);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, moe_gather_kernel, x, xdt, (int64_t)K, per_slot ? 1 : (int)top_k,
                               (const int*)(L.offsets + n_expert), (const int*)L.rows, (int64_t)entries, L.xg,
                               L.xscale) != cudaSuccess)
            return GGUF_ERR_CUDA;
    }
    return grouped_gemm_run(w_experts, qtype, n_expert, N, K, L.xg, L.xscale, entries, L.tiles, L.ntiles, L.offsets,
                            L.rows, L.max_tiles, residual, y, ydt, status, stream, pdl);
}

}  // namespace gg
