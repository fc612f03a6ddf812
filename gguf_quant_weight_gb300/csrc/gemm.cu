// Tensor-core GEMMs on tcgen05 (sm_103a).
//
// Swap-AB form: the weight is UMMA operand A (M = 128 weight rows per CTA,
// K-major) and the activations are operand B (N = BN token rows, K-major), so a
// tile is 128 output features x BN tokens accumulated in f32 in TMEM (128 lanes
// x BN columns).  Both operands sit in shared memory in the 128-byte-swizzled
// K-major layout (8-row x 128-byte atoms), K advancing 64 values per stage.
//
// Warp roles in one CTA:
//   warp 0        TMA producer (one elected lane)
//   warp 1        TMEM allocation and MMA issue (one elected lane)
//   warps 2..     A-operand producers when the weight is decoded in the kernel
//                 (gemm_fused.cu), then the epilogue: TMEM -> registers,
//                 + residual, round, store.
// Every wait is a bounded mbarrier poll; a timeout is recorded in the status
// word and the kernel still releases its TMEM before returning.
//
// This file holds the dense kernel used on a decoded weight buffer (ROCm
// llama.cpp PR #37 "one-time K-padded f16 dequantization for prefill GEMMs",
// "How it works": decode once into a K-padded buffer, then a plain GEMM with
// the padded leading dimension) and the activation conversion pass.
#include <mutex>

#include "tc_gemm.cuh"

namespace gg {

// ------------------------------------------------------------------ activation conversion

namespace {

// Activation rows to 16 bits.  For an f16 copy the row is scaled by 2^-s
// first, with s = floor(log2(max |x|)) - 14, so that its largest magnitude
// lands in [2^14, 2^15): a bf16 or f32 row whose values exceed f16's range
// (65504) or sit below its normal range (2^-14) keeps its 8 (bf16) or 11
// (f32, rounded) significant bits instead of turning into inf or losing bits
// in f16 subnormals.  The scale 2^s goes to scale[m]; the GEMM's epilogue
// multiplies row m's sums by it.  A power of two is exact, so rows already in
// range give the same result bit for bit as an unscaled copy.  (A row holding
// inf or NaN is left unscaled: those values pass through as they are.)  A
// bf16 copy keeps f32's range and is never scaled.
template <int XDT>
__device__ __forceinline__ void load8(const void* x, int64_t off, float v[8]) {
    if (XDT == GGUF_DT_F32) {
        const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + off);
        const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(x) + off + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
        const uint4 t = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + off);
        const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t lo = w4[j] & 0xFFFFu, hi = w4[j] >> 16;
            if (XDT == GGUF_DT_BF16) { v[2 * j] = __uint_as_float(lo << 16); v[2 * j + 1] = __uint_as_float(hi << 16); }
            else { v[2 * j] = f16_bits_to_float(lo); v[2 * j + 1] = f16_bits_to_float(hi); }
        }
    }
}

// One CTA of 256 threads per activation row (rows strided over the grid).
// Each thread loads its chunks of 8 values -- up to RCH of them, so a row of up
// to 256 * 8 * RCH values is read once and held in registers with every load
// in flight -- the CTA reduces the row's largest finite magnitude, and the
// threads convert their chunks from registers.  Longer rows take a second
// pass over global memory.
constexpr int kConvThreads = 256, kConvChunks = 8;

template <int XDT>
__global__ void __launch_bounds__(kConvThreads) convert_rows_kernel(const void* __restrict__ x, int64_t M, int64_t K,
                                                                    uint16_t* __restrict__ out, int odt_bf16,
                                                                    float* __restrict__ scale,
                                                                    uint32_t* __restrict__ zero, int nzero) {
    __shared__ float red_max[kConvThreads / 32];
    __shared__ int red_fin[kConvThreads / 32];
    // the fused GEMM after this kernel may start now (its weight stream and
    // decoding need nothing from here; what reads these outputs waits first)
    pdl_launch_dependents();
    // the GEMM that follows on the stream counts on these words being zero
    if (blockIdx.x == 0)
        for (int j = threadIdx.x; j < nzero; j += blockDim.x) zero[j] = 0u;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t nch = K / 8;                                  // chunks of 8 values in a row
    const bool in_regs = nch <= (int64_t)kConvThreads * kConvChunks;
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const int64_t base = m * K;
        float v[kConvChunks][8];
        float amax = 0.f;   // largest finite magnitude; a non-finite value marks the row
        bool finite = true;
        if (in_regs) {
#pragma unroll
            for (int c = 0; c < kConvChunks; ++c) {
                const int64_t ch = tid + (int64_t)c * kConvThreads;
                if (ch < nch) load8<XDT>(x, base + 8 * ch, v[c]);
            }
#pragma unroll
            for (int c = 0; c < kConvChunks; ++c) {
                if (tid + (int64_t)c * kConvThreads < nch) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        finite = finite && isfinite(v[c][j]);
                        amax = fmaxf(amax, fabsf(v[c][j]));
                    }
                }
            }
        } else {
            for (int64_t ch = tid; ch < nch; ch += kConvThreads) {
                float t[8];
                load8<XDT>(x, base + 8 * ch, t);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    finite = finite && isfinite(t[j]);
                    amax = fmaxf(amax, fabsf(t[j]));
                }
            }
        }
        float mul = 1.f, back = 1.f;
        if (!odt_bf16) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const bool wf = __all_sync(0xffffffffu, finite);
            if (lane == 0) { red_max[warp] = amax; red_fin[warp] = wf ? 1 : 0; }
            __syncthreads();
            amax = 0.f;
            finite = true;
#pragma unroll
            for (int w = 0; w < kConvThreads / 32; ++w) {
                amax = fmaxf(amax, red_max[w]);
                finite = finite && red_fin[w];
            }
            __syncthreads();   // red_* reused by the next row
            if (finite && amax > 0.f) {
                const int s = max(-100, min(100, ilogbf(amax) - 14));
                mul = ldexpf(1.f, -s);
                back = ldexpf(1.f, s);
            }
        }
        auto store8 = [&](int64_t ch, const float (&t)[8]) {
            uint16_t o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                o[j] = odt_bf16 ? __bfloat16_as_ushort(__float2bfloat16_rn(t[j]))
                                : __half_as_ushort(__float2half_rn(t[j] * mul));
            *reinterpret_cast<uint4*>(out + base + 8 * ch) =
                make_uint4(o[0] | (uint32_t)o[1] << 16, o[2] | (uint32_t)o[3] << 16, o[4] | (uint32_t)o[5] << 16,
                           o[6] | (uint32_t)o[7] << 16);
        };
        if (in_regs) {
#pragma unroll
            for (int c = 0; c < kConvChunks; ++c) {
                const int64_t ch = tid + (int64_t)c * kConvThreads;
                if (ch < nch) store8(ch, v[c]);
            }
        } else {
            for (int64_t ch = tid; ch < nch; ch += kConvThreads) {
                float t[8];
                load8<XDT>(x, base + 8 * ch, t);
                store8(ch, t);
            }
        }
        if (tid == 0 && scale) scale[m] = back;
    }
}

}  // namespace

cudaError_t convert_activations(const void* x, int xdt, int64_t M, int64_t K, void* out, int odt, float* scale,
                                int num_sms, cudaStream_t s, uint32_t* zero, int nzero) {
    if (K % 8 != 0) return cudaErrorInvalidValue;
    const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(M, (int64_t)num_sms * 8));
    const int bf = odt == GGUF_DT_BF16 ? 1 : 0;
    uint16_t* o = static_cast<uint16_t*>(out);
    if (xdt == GGUF_DT_F32)
        convert_rows_kernel<GGUF_DT_F32><<<(unsigned)blocks, kConvThreads, 0, s>>>(x, M, K, o, bf, scale, zero, nzero);
    else if (xdt == GGUF_DT_F16)
        convert_rows_kernel<GGUF_DT_F16><<<(unsigned)blocks, kConvThreads, 0, s>>>(x, M, K, o, bf, scale, zero, nzero);
    else
        convert_rows_kernel<GGUF_DT_BF16><<<(unsigned)blocks, kConvThreads, 0, s>>>(x, M, K, o, bf, scale, zero, nzero);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

int make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t inner,
                 uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return GGUF_ERR_CUDA;
    (void)elem_bytes;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t es[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GGUF_OK : GGUF_ERR_UNSUPPORTED;
}

// ------------------------------------------------------------------ dense kernel

namespace {

template <int BN>
__global__ void __launch_bounds__(192, 1)
    dense_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const TcEpilogue ep, int nk, int ab_bf16, int* status) {
    using C = TcCfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = align_up_1024(smem_raw);
    uint8_t* sA = base;
    uint8_t* sB = base + C::S * C::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + C::S * C::B_BYTES);
    uint64_t* empty = full + C::S;
    uint64_t* tfull = empty + C::S;
    uint32_t* tslot = reinterpret_cast<uint32_t*>(tfull + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * 128, t0 = blockIdx.y * BN;
    __shared__ float s_xscale[BN];   // the tile's activation-row scales, for the epilogue
    for (int i = threadIdx.x; i < BN; i += blockDim.x)
        s_xscale[i] = (ep.xscale && t0 + i < ep.M) ? ep.xscale[t0 + i] : 1.f;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::S; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        mbar_init(tfull, 1);
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tslot, C::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % C::S;
            const uint32_t ph = (uint32_t)((kb / C::S) & 1);
            if (!mbar_wait(&empty[s], ph ^ 1, status)) break;
            mbar_arrive_expect_tx(&full[s], C::A_BYTES + C::B_BYTES);
            tma_load_2d(sA + s * C::A_BYTES, &tmA, kb * 64, n0, &full[s]);
            tma_load_2d(sB + s * C::B_BYTES, &tmB, kb * 64, t0, &full[s]);
        }
    } else if (warp == 1 && lane == 0) {
        const uint32_t idesc = idesc_f16(128, BN, ab_bf16);
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % C::S;
            const uint32_t ph = (uint32_t)((kb / C::S) & 1);
            if (!mbar_wait(&full[s], ph, status)) break;
            tc_fence_after();
            const uint32_t a0 = smem_u32(sA + s * C::A_BYTES), b0 = smem_u32(sB + s * C::B_BYTES);
#pragma unroll
            for (int k = 0; k < 4; ++k)
                umma_f16(tmem, sw128_desc(a0 + 32 * k), sw128_desc(b0 + 32 * k), idesc, (kb | k) != 0);
            umma_commit(&empty[s]);
        }
        umma_commit(tfull);
    } else if (warp >= 2) {
        if (mbar_wait(tfull, 0, status)) {
            tc_fence_after();
            tc_epilogue<BN>(ep, tmem, warp & 3, lane, n0, t0, s_xscale);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int BN>
cudaError_t launch_dense(const CUtensorMap& a, const CUtensorMap& b, const TcEpilogue& ep, int nk, int ab_bf16,
                         int* status, cudaStream_t s) {
    using C = TcCfg<BN>;
    auto k = dense_tc_kernel<BN>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)ceil_div(ep.N, 128), (unsigned)ceil_div(ep.M, BN));
    k<<<grid, 192, C::SMEM, s>>>(a, b, ep, nk, ab_bf16, status);
    return cudaGetLastError();
}

}  // namespace

int pick_bn(int64_t N, int64_t M, int num_sms) {
    int best = 256;
    double best_cost = 1e30;
    for (int bn : {256, 128, 64, 32}) {
        const int64_t tiles = ceil_div(N, 128) * ceil_div(M, bn);
        const double cost = (double)ceil_div(tiles, num_sms) * (bn + 64);
        if (cost < best_cost - 1e-9) { best_cost = cost; best = bn; }
    }
    return best;
}

size_t dense_workspace_bytes(int64_t N, int64_t K, int64_t M) {
    (void)N;
    return (size_t)(act_copy_bytes(M, K) + act_scale_bytes(M));   // converted activations, then their row scales
}

int dense_gemm_run(const void* wdense, int wdt, int64_t ld, int64_t N, int64_t K, const void* x, int xdt, int64_t M,
                   const void* residual, void* y, int ydt, void* workspace, int num_sms, int* status,
                   cudaStream_t stream) {
    if (N > (int64_t)INT32_MAX || M > (int64_t)INT32_MAX) return GGUF_ERR_UNSUPPORTED;
    const void* xb = x;
    float* xscale = nullptr;
    if (xdt != wdt) {
        xscale = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + act_copy_bytes(M, K));
        if (convert_activations(x, xdt, M, K, workspace, wdt, xscale, num_sms, stream) != cudaSuccess)
            return GGUF_ERR_CUDA;
        xb = workspace;
    }
    const CUtensorMapDataType dt = wdt == GGUF_DT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const int bn = pick_bn(N, M, num_sms);
    CUtensorMap ta, tb;
    int st = make_tmap_2d(&ta, wdense, dt, 2, (uint64_t)K, (uint64_t)N, (uint64_t)ld * 2, 64, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != GGUF_OK) return st;
    st = make_tmap_2d(&tb, xb, dt, 2, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2, 64, (uint32_t)bn,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != GGUF_OK) return st;
    TcEpilogue ep{residual, y, ydt, N, M, xscale};
    const int nk = (int)(K / 64), bf = wdt == GGUF_DT_BF16 ? 1 : 0;
    cudaError_t e;
    switch (bn) {
        case 256: e = launch_dense<256>(ta, tb, ep, nk, bf, status, stream); break;
        case 128: e = launch_dense<128>(ta, tb, ep, nk, bf, status, stream); break;
        case 64: e = launch_dense<64>(ta, tb, ep, nk, bf, status, stream); break;
        default: e = launch_dense<32>(ta, tb, ep, nk, bf, status, stream); break;
    }
    return e == cudaSuccess ? GGUF_OK : GGUF_ERR_CUDA;
}

}  // namespace gg

namespace gg {

// ------------------------------------------------------------------ allocation-free variant of the dense GEMM
//
// Some callers hand this library only their input and output buffers and may
// not obtain device memory at all: code embedded in a host program that owns
// every device allocation through its own fixed pool, or code running where a
// cudaMalloc would implicitly synchronize the device and stall the other work
// in flight.  For them gguf_dense_gemm_noalloc keeps its scratch (the
// activations converted to the weight's 16-bit type) in the array below, which
// is part of this library's device image: every GPU that loads the library
// holds these 8 MiB until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) uint8_t g_dense_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mu;
void* g_noalloc_scratch_ptr[64];

// In host code the array's name is only a host-side stand-in; the device
// address is looked up once per device, with that device current.
int noalloc_scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return GGUF_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_dense_noalloc_scratch) != cudaSuccess || p == nullptr) return GGUF_ERR_CUDA;
        g_noalloc_scratch_ptr[dev] = p;
    }
    *out = g_noalloc_scratch_ptr[dev];
    return GGUF_OK;
}

}  // namespace

}  // namespace gg

extern "C" int gguf_dense_gemm_noalloc(const void* wdense, int wdt, int64_t ld, int64_t N, int64_t K, const void* x,
                                       int xdt, int64_t M, const void* residual, void* y, int ydt,
                                       gguf_stream_t stream) {
    using namespace gg;
    if (!wdense || !x || !y || N <= 0 || K <= 0 || M <= 0) return GGUF_ERR_INVALID_ARG;
    if ((wdt != GGUF_DT_F16 && wdt != GGUF_DT_BF16) || (xdt != GGUF_DT_F16 && xdt != GGUF_DT_BF16) ||
        (ydt != GGUF_DT_F32 && ydt != GGUF_DT_F16 && ydt != GGUF_DT_BF16))
        return GGUF_ERR_UNSUPPORTED;
    if (K % 64 != 0 || ld < K || ld % 8 != 0) return GGUF_ERR_INVALID_ARG;
    auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (!a16(wdense) || !a16(x) || !a16(y) || (residual && !a16(residual))) return GGUF_ERR_MISALIGNED;
    // the converted activations must fit the built-in scratch: M * K * 2 bytes <= 8 MiB
    if (M > (int64_t)(kNoAllocScratchBytes / 2) || dense_workspace_bytes(N, K, M) > kNoAllocScratchBytes)
        return GGUF_ERR_WORKSPACE;
    int num_sms = 0;
    int* status = nullptr;
    int st = current_device_launch_facts(&num_sms, &status);
    if (st != GGUF_OK) return st;
    void* scratch = nullptr;
    if ((st = noalloc_scratch_address(&scratch)) != GGUF_OK) return st;
    return dense_gemm_run(wdense, wdt, ld, N, K, x, xdt, M, residual, y, ydt, scratch, num_sms, status,
                          (cudaStream_t)stream);
}
