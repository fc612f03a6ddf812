// Q6_K plane regrouping and its inverse (OpenVINO PR #39119 "FullyConnectedGGUF",
// "Transformation": Q6_K blocks are regrouped once into aligned planes
// QL[nblk][128] | QH[nblk][64] | SC[nblk][16] | D[nblk]; same size, same bytes).
//
// One CTA moves a tile of 64 blocks (13,440 bytes, a multiple of 16): the
// contiguous side (the raw blocks) moves with 16-byte global accesses, the
// scattered side goes through shared memory.  Every plane segment of a full
// tile starts on a 16-byte boundary, so both sides use 16-byte global
// accesses; a partial last tile moves byte by byte.
#include "common.cuh"

namespace gg {

namespace {

constexpr int kTileBlocks = 64;
constexpr int kTileBytes = kTileBlocks * 210;
constexpr int kThreads = 256;

// Field f of block-in-tile b: (offset inside the 210-byte block, bytes).
__device__ __forceinline__ void field_geom(int f, int& off, int& len) {
    off = f == 0 ? 0 : f == 1 ? 128 : f == 2 ? 192 : 208;
    len = f == 0 ? 128 : f == 1 ? 64 : f == 2 ? 16 : 2;
}

__global__ void __launch_bounds__(kThreads) q6k_planes_kernel(const uint8_t* __restrict__ src,
                                                              uint8_t* __restrict__ dst, int64_t nblk,
                                                              int inverse) {
    __shared__ __align__(16) uint8_t tile[kTileBytes];
    const int64_t b0 = (int64_t)blockIdx.x * kTileBlocks;
    const int nb = (int)(nblk - b0 < kTileBlocks ? nblk - b0 : (int64_t)kTileBlocks);
    const bool full = nb == kTileBlocks;
    const int64_t plane_off[4] = {0, 128 * nblk, 192 * nblk, 208 * nblk};

    if (!inverse) {
        // raw blocks -> tile (contiguous)
        const uint8_t* s = src + b0 * 210;
        if (full) {
            for (int i = threadIdx.x; i < kTileBytes / 16; i += kThreads)
                reinterpret_cast<uint4*>(tile)[i] = __ldg(reinterpret_cast<const uint4*>(s) + i);
        } else {
            for (int i = threadIdx.x; i < nb * 210; i += kThreads) tile[i] = s[i];
        }
        __syncthreads();
        // tile -> four plane segments
        for (int f = 0; f < 4; ++f) {
            int off, len;
            field_geom(f, off, len);
            uint8_t* d = dst + plane_off[f] + b0 * len;
            const int seg = nb * len;
            if (full) {
                for (int q = threadIdx.x; q < seg / 16; q += kThreads) {
                    uint16_t h[8];
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int byte = q * 16 + 2 * t;  // byte inside the segment
                        h[t] = *reinterpret_cast<const uint16_t*>(tile + (byte / len) * 210 + off + byte % len);
                    }
                    uint4 v;
                    v.x = h[0] | (uint32_t)h[1] << 16; v.y = h[2] | (uint32_t)h[3] << 16;
                    v.z = h[4] | (uint32_t)h[5] << 16; v.w = h[6] | (uint32_t)h[7] << 16;
                    reinterpret_cast<uint4*>(d)[q] = v;
                }
            } else {
                for (int byte = threadIdx.x; byte < seg; byte += kThreads)
                    d[byte] = tile[(byte / len) * 210 + off + byte % len];
            }
        }
    } else {
        // four plane segments -> tile (block layout)
        for (int f = 0; f < 4; ++f) {
            int off, len;
            field_geom(f, off, len);
            const uint8_t* s = src + plane_off[f] + b0 * len;
            const int seg = nb * len;
            if (full) {
                for (int q = threadIdx.x; q < seg / 16; q += kThreads) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(s) + q);
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        const int byte = q * 16 + 2 * t;
                        *reinterpret_cast<uint16_t*>(tile + (byte / len) * 210 + off + byte % len) =
                            (uint16_t)(w[t >> 1] >> (16 * (t & 1)));
                    }
                }
            } else {
                for (int byte = threadIdx.x; byte < seg; byte += kThreads)
                    tile[(byte / len) * 210 + off + byte % len] = s[byte];
            }
        }
        __syncthreads();
        uint8_t* d = dst + b0 * 210;
        if (full) {
            for (int i = threadIdx.x; i < kTileBytes / 16; i += kThreads)
                reinterpret_cast<uint4*>(d)[i] = reinterpret_cast<const uint4*>(tile)[i];
        } else {
            for (int i = threadIdx.x; i < nb * 210; i += kThreads) d[i] = tile[i];
        }
    }
}

}  // namespace

cudaError_t repack_q6k_launch(const void* src, void* dst, int64_t nblk, int inverse, cudaStream_t stream) {
    const int64_t tiles = ceil_div(nblk, kTileBlocks);
    q6k_planes_kernel<<<(unsigned)tiles, kThreads, 0, stream>>>(static_cast<const uint8_t*>(src),
                                                                  static_cast<uint8_t*>(dst), nblk, inverse);
    return cudaGetLastError();
}

}  // namespace gg
