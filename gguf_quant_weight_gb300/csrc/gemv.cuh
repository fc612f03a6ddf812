// Host-visible parameters of the decode GEMV kernel.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <algorithm>

namespace gg {

struct GemvParams {
    const uint8_t* w;
    int qtype, layout;
    int64_t N, K;
    const void* x;
    int xdt, M;
    const void* residual;
    void* y;
    int ydt;
    int* status;
    int pdl;               // launch with programmatic stream serialization
    void* act_image;       // workspace: the quantized activations (codes + per-block entries)
    int direct;            // unit fields 16-byte aligned: load straight into registers
    int tile;              // rows staged whole in shared memory, two CTAs per SM: 1 tile, 2 pair, 3 row-lane kernel
    int force;             // -1: the plan's choice; else one of the GEMV_* kernels (test hook)
    int cluster;           // row-lane kernel: CTAs per cluster sharing the activation quantization (1, 2, 4)
    // plan (filled by gemv_plan)
    int64_t rb;            // bytes per weight row (raw layout)
    int64_t rows_per_cta;  // rows owned by one CTA
    int chunk_rows;        // rows per staged chunk
    int stages;            // chunk buffers in shared memory
    int64_t stage_bytes;
    // routed mode (the MoE decode form of the staged kernel): grid.y runs over
    // the routed rows; row r multiplies activation row r / route_div of the
    // image (img_rows rows) against the expert ids[r] of n_expert (w holds the
    // experts' [N, rb] blocks back to back) and writes output row r
    const int32_t* ids;
    int64_t n_expert;
    int route_div;
    int64_t img_rows;
    // test-only dumps (nullptr in production)
    int8_t* dbg_qa;
    float* dbg_da;
    int32_t* dbg_s;
    int32_t* dbg_D;
};

// GEMV kernels a plan can choose (ids reported by the test hooks).
enum { GEMV_STAGED = 0, GEMV_DIRECT = 1, GEMV_TILE = 2, GEMV_PAIR = 3, GEMV_ROWLANE = 4 };
// The kernel a filled plan launches.
int gemv_kind(const GemvParams& p);

// Fills the plan fields; returns GGUF_OK or GGUF_ERR_UNSUPPORTED when the
// activations and one chunk do not fit in max_smem bytes of shared memory.
int gemv_plan(GemvParams& p, int num_sms, int max_smem, int* grid, size_t* smem);
// Workspace bytes of a GEMV call (the quantized activation image).
size_t gemv_workspace_bytes(int64_t M, int64_t K);
cudaError_t gemv_launch(const GemvParams& p, int grid, size_t smem, bool dump, cudaStream_t stream);

// MoE decode form (a few routed rows, Q4_K / Q5_K): every routed row p =
// token * top_k + slot is a GEMV of its activation row (x[token], or x[p] in the
// per-slot form) against expert ids[p]'s blocks, on the int8 path.
struct MoeMvParams {
    const uint8_t* w;       // expert weights back to back: [E * N, rb]
    int qtype;
    int64_t n_expert, N, K, rb;
    const int32_t* ids;     // [entries]
    int entries, top_k, per_slot;
    const void* x;          // activation rows [T, K] (per-slot form: [T * top_k, K])
    int xdt;
    const uint8_t* image;   // workspace for their act_quant image (more than a few routed rows)
    int64_t rows;           // activation rows: T, or T * top_k in the per-slot form
    const void* residual;
    void* y;
    int ydt;
    int* status;
    int pdl;                // the GEMV as a dependent launch of the quantizer (other formats)
    // test hook (a separate instantiation): routed row p's activation codes
    // [p][K], scales and sums [p][K/32], sub-block dots [p][N][K/32]
    int8_t* dbg_qa;
    float* dbg_da;
    int32_t* dbg_s;
    int32_t* dbg_D;
};
size_t moe_mv_image_bytes(int64_t rows, int64_t K);
cudaError_t moe_mv_launch(const MoeMvParams& mp, cudaStream_t stream, bool dump = false);
// The decode form for the other formats: the activation rows quantized once,
// then the staged GEMV kernel in routed mode (one grid row per routed row).
int moe_mv_staged_run(const MoeMvParams& mp, int num_sms, int max_smem, cudaStream_t stream);

}  // namespace gg
