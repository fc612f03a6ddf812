// Decode-once into a K-padded f16/bf16 buffer (ROCm llama.cpp PR #37 "one-time
// K-padded f16 dequantization for prefill GEMMs", "How it works": the weight is
// decoded a single time into a buffer whose row stride is padded by one cache
// line, and the dense GEMM then reads it with that leading dimension;
// "Correctness": the padding changes only the stride).
//
// One thread writes 8 consecutive outputs (one 16-byte store); pad columns are
// written as zero.  This runs once per weight, so it is kept simple: it is a
// plain HBM-bound stream (read the blocks, write 2 bytes per value).
#include "formats.cuh"

namespace gg {

namespace {

template <int QT, bool PLANES>
__global__ void dequant_padded_kernel(const uint8_t* __restrict__ w, int64_t N, int64_t K, int64_t ld,
                                      void* __restrict__ out, int odt) {
    const int64_t per_row = ld / 8;
    const int64_t total = N * per_row;
    const int64_t rb = K / block_values(QT) * block_bytes(QT);
    const int64_t nblk = N * (K / 256);
    for (int64_t item = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; item < total;
         item += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = item / per_row;
        const int64_t k0 = (item % per_row) * 8;
        float v[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int64_t k = k0 + t;
            if (k >= K) { v[t] = 0.f; continue; }
            const int64_t kb = k / block_values(QT);
            const int e = (int)(k % block_values(QT));
            if (PLANES) v[t] = decode_q6k_planes_elem(w, nblk, n * (K / 256) + kb, e);
            else v[t] = decode_elem<QT>(w + n * rb + kb * block_bytes(QT), e);
        }
        uint32_t packed[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            uint16_t a, b;
            if (odt == GGUF_DT_F16) {
                a = __half_as_ushort(__float2half_rn(v[2 * t]));
                b = __half_as_ushort(__float2half_rn(v[2 * t + 1]));
            } else {
                a = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * t]));
                b = __bfloat16_as_ushort(__float2bfloat16_rn(v[2 * t + 1]));
            }
            packed[t] = (uint32_t)a | ((uint32_t)b << 16);
        }
        reinterpret_cast<uint4*>(out)[item] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
}

template <int QT, bool PLANES>
cudaError_t go(const void* w, int64_t N, int64_t K, int64_t ld, void* out, int odt, int num_sms,
               cudaStream_t s) {
    const int64_t total = N * (ld / 8);
    const int64_t blocks = std::min<int64_t>(ceil_div(total, 256), (int64_t)num_sms * 16);
    dequant_padded_kernel<QT, PLANES><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const uint8_t*>(w), N, K, ld,
                                                                        out, odt);
    return cudaGetLastError();
}

}  // namespace

cudaError_t dequant_padded_launch(const void* w, int qtype, int layout, int64_t N, int64_t K, void* out, int odt,
                                  int64_t ld, int num_sms, cudaStream_t s) {
    switch (qtype) {
        case GGUF_Q4_0: return go<GGUF_Q4_0, false>(w, N, K, ld, out, odt, num_sms, s);
        case GGUF_Q4_1: return go<GGUF_Q4_1, false>(w, N, K, ld, out, odt, num_sms, s);
        case GGUF_Q5_0: return go<GGUF_Q5_0, false>(w, N, K, ld, out, odt, num_sms, s);
        case GGUF_Q5_1: return go<GGUF_Q5_1, false>(w, N, K, ld, out, odt, num_sms, s);
        case GGUF_Q8_0: return go<GGUF_Q8_0, false>(w, N, K, ld, out, odt, num_sms, s);
        case GGUF_Q2_K: return go<GGUF_Q2_K, false>(w, N, K, ld, out, odt, num_sms, s);
        case GGUF_Q3_K: return go<GGUF_Q3_K, false>(w, N, K, ld, out, odt, num_sms, s);
        case GGUF_Q4_K: return go<GGUF_Q4_K, false>(w, N, K, ld, out, odt, num_sms, s);
        case GGUF_Q5_K: return go<GGUF_Q5_K, false>(w, N, K, ld, out, odt, num_sms, s);
        case GGUF_Q6_K:
            return layout == GGUF_LAYOUT_Q6K_PLANES ? go<GGUF_Q6_K, true>(w, N, K, ld, out, odt, num_sms, s)
                                                    : go<GGUF_Q6_K, false>(w, N, K, ld, out, odt, num_sms, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gg
