// Pieces shared by the tcgen05 GEMM kernels: tile configuration, tensor maps,
// the TMEM -> global epilogue with the fused residual Add.
#pragma once
#include "tc.cuh"
#include "gemm.cuh"

namespace gg {

// Tile of 128 weight rows x BN tokens, K step 64 (one 128-byte swizzle atom of f16).
template <int BN>
struct TcCfg {
    static constexpr int A_BYTES = 128 * 64 * 2;   // 16 KB
    static constexpr int B_BYTES = BN * 64 * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int S = (196608 / STAGE) > 8 ? 8 : (196608 / STAGE);
    static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
    static constexpr int SMEM = S * STAGE + 1024 + 256;
};

struct TcEpilogue {
    const void* residual;  // [M][N] of ydt or null
    void* y;               // [M][N]
    int ydt;
    int64_t N, M;          // output features, tokens
    const float* xscale;   // [M] power-of-two scale of each activation row's f16 copy, or null (1)
};

__device__ __forceinline__ uint8_t* align_up_1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Warp q (0..3) of the epilogue reads TMEM lanes 32q..32q+31 (weight rows
// n0 + 32q + lane) for all BN token columns, adds the residual and stores.
// xs: the BN activation-row scales of the tile, staged in shared memory.
template <int BN>
__device__ __forceinline__ void tc_epilogue(const TcEpilogue& ep, uint32_t tmem, int q, int lane, int64_t n0,
                                            int64_t t0, const float* xs) {
    const int64_t n = n0 + 32 * q + lane;
#pragma unroll 1
    for (int c = 0; c < BN / 16; ++c) {
        uint32_t v[16];
        tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 16 * c, v);
        tmem_ld_wait();
        if (n < ep.N) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int64_t m = t0 + 16 * c + j;
                if (m < ep.M) {
                    float o = __uint_as_float(v[j]);
                    o *= xs[16 * c + j];
                    if (ep.residual) o += load_act(ep.residual, ep.ydt, m * ep.N + n);
                    store_out(ep.y, ep.ydt, m * ep.N + n, o);
                }
            }
        }
    }
}

int make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, uint64_t inner,
                 uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                 CUtensorMapSwizzle swz);
// X [M, K] (F32/F16/BF16) -> odt (F16/BF16) into out, row by row; an F16 copy
// of row m holds x * 2^-s_m (scale[m] = 2^s_m, see the kernel), a BF16 copy x
// itself (scale[m] = 1).  scale may be null.  Also zeroes nzero 32-bit words at
// `zero` (the split-K tickets of the GEMM that follows).  K % 8 == 0.
cudaError_t convert_activations(const void* x, int xdt, int64_t M, int64_t K, void* out, int odt, float* scale,
                                int num_sms, cudaStream_t s, uint32_t* zero = nullptr, int nzero = 0);
// Bytes of the activation copy that precedes the row scales in a workspace.
__host__ __device__ inline int64_t act_copy_bytes(int64_t M, int64_t K) { return (M * K * 2 + 255) / 256 * 256; }
__host__ __device__ inline int64_t act_scale_bytes(int64_t M) { return (M * 4 + 255) / 256 * 256; }
int pick_bn(int64_t N, int64_t M, int num_sms);

}  // namespace gg
