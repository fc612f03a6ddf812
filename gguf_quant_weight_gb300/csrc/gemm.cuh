// Host entry points of the tensor-core GEMMs (fused decode-in-smem, and dense
// on a decoded buffer).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <stddef.h>

namespace gg {

// Workspace of the fused GEMM on a device with num_sms SMs: the F16
// activations, plus the split-K partial sums and tickets when the plan for
// that SM count splits K.
size_t gemm_workspace_bytes(int qtype, int64_t N, int64_t K, int64_t M, int num_sms);
size_t dense_workspace_bytes(int64_t N, int64_t K, int64_t M);

// pdl: launch the GEMM as a programmatic dependent of its activation
// conversion kernel (overlaps its start with the conversion)
int gemm_fused_run(const void* w, int qtype, int layout, int64_t N, int64_t K, const void* x, int xdt, int64_t M,
                   const void* residual, void* y, int ydt, void* workspace, int num_sms, int* status,
                   cudaStream_t stream, int pdl);

int dense_gemm_run(const void* wdense, int wdt, int64_t ld, int64_t N, int64_t K, const void* x, int xdt, int64_t M,
                   const void* residual, void* y, int ydt, void* workspace, int num_sms, int* status,
                   cudaStream_t stream);

// Grouped (MoE) form of the fused GEMM: work items (expert, token tile) and
// the grouped activation rows come from the routing kernel (moe.cu).
int grouped_gemm_run(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K, const void* xg,
                     const float* xscale, int64_t rows_cap, const int4* tiles, const int* ntiles, const int* offsets,
                     const int* rows, int64_t max_tiles, const void* residual, void* y, int ydt, int* status,
                     cudaStream_t stream, int pdl = 0);

// Launch facts of the current device (SM count, device address of the status
// word), as the C entry points use them.
int current_device_launch_facts(int* num_sms, int** status);

}  // namespace gg
