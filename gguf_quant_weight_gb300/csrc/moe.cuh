// Host entry points of the MoE expert GEMM (mul_mm_id).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

namespace gg {

// At most this many routed rows (T * top_k) take the decode form (one int8
// GEMV per routed row, no routing): 128 for Q4_K, Q5_K, Q2_K, Q3_K and Q6_K,
// 32 for Q4_0, Q4_1, Q5_0 and Q5_1, 16 for Q8_0 (where the routed tensor-core
// path measured faster above that on 128 experts of 768 x 2048, top-8).
constexpr int kMoeMvRows = 128;
int moe_mv_max_rows(int qtype);
// The batch-size rule (and its GGUF_MM_MOE_MV=0 override): does this many
// routed rows of qtype experts take the decode form?  Host only, no CUDA call.
bool moe_decode_form(int qtype, int64_t entries);

size_t moe_workspace_bytes(int qtype, int64_t n_expert, int64_t N, int64_t K, int64_t T, int64_t top_k);

// Integer intermediates of the decode form (test hook): routed row p's
// activation codes [p][K], scales and sums [p][K/32], dots [p][N][K/32].
struct MoeMvDump {
    int8_t* qa;
    float* da;
    int32_t* s;
    int32_t* D;
};

// dump: run the decode form with its integer terms written out
// (GGUF_ERR_UNSUPPORTED when this batch does not take the decode form).
// pdl: chain the routed path's gather and grouped GEMM as programmatic
// dependent launches (each waits before reading the kernel before it).
// form: -1 the batch-size rule (moe_mv_max_rows), 0 the routed tensor-core
// path, 1 the decode form (GGUF_ERR_UNSUPPORTED above kMoeMvRows routed rows).
int moe_run(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K, const void* x, int xdt,
            int64_t T, const int32_t* ids, int64_t top_k, const void* residual, void* y, int ydt, void* workspace,
            int num_sms, int* status, cudaStream_t stream, bool per_slot = false, const MoeMvDump* dump = nullptr,
            int pdl = 0, int form = -1);

// The routing step alone (test hook): per-expert group offsets [E + 1], the
// number of (expert, token tile) work items, the items {expert, first row,
// rows, 0} (at most max_tiles) and the grouped entry list [entries].
int moe_route_debug(const int32_t* ids, int64_t entries, int64_t n_expert, int* offsets, int* ntiles, int4* tiles,
                    int64_t max_tiles, int* rows, cudaStream_t stream);
// Work items the routing step can produce for this many experts and routed rows.
int64_t moe_max_tiles(int64_t n_expert, int64_t entries);

}  // namespace gg
