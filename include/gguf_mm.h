/*
 * gguf_mm.h -- C ABI of libgguf_mm.so: matrix multiplication run directly on
 * GGUF block-quantized weights on one NVIDIA GB300 (sm_103a).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is DEVICE memory owned by the caller, unless the
 *    argument says otherwise.  The library never frees, retains or caches a
 *    caller pointer past the call.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and the call returns without a host synchronisation.  A returned
 *    GGUF_OK means the work was validated and launched; device-side failures
 *    (a bounded wait that expired) are reported later by gguf_mm_check_errors().
 *  - Matrices are row-major and contiguous.  X is [M, K], Y is [M, N]; the
 *    optional residual has Y's dtype and shape and may alias Y.
 *  - A weight tensor W[N, K] stays in GGUF byte blocks: row n is the K/blk
 *    blocks covering W[n, 0..K) back to back, i.e. a [N, K/blk*block_bytes] u8
 *    array (OpenVINO PR #39119 "FullyConnectedGGUF", "Why a new primitive").
 *  - Block structs (GGUF on-disk layout; GGUF Support Proposal for mobius,
 *    sections 1.2 and 7): Q4_0 18 B / 32 values {d f16, qs[16]}, w = (q-8)*d;
 *    Q4_1 20 B {d, m f16, qs[16]}, w = q*d + m; Q5_0 22 B {d, qh[4], qs[16]},
 *    w = (q5-16)*d; Q5_1 24 B {d, m, qh[4], qs[16]}, w = q5*d + m (element
 *    e < 16 in the low nibble of qs[e], e >= 16 in the high nibble of
 *    qs[e-16], its fifth bit bit e of the little-endian qh word);
 *    Q8_0 34 B / 32 values {d f16, qs[32] i8}, w = d*q;
 *    Q2_K 84 B / 256 {scales[16], qs[64], d, dmin f16}, w = d*(sc&15)*q2 -
 *    dmin*(sc>>4) per 16-value sub-block; Q3_K 110 B / 256 {hmask[32], qs[64],
 *    scales[12], d f16}, w = d*(scale6 - 32)*q3 with q3 = q2 - 4 where the
 *    element's hmask bit is clear (element 128h + 32j + 16p + l: bits 2j..2j+1
 *    of qs[32h + 16p + l]; hmask bit e/32 of byte e%32);
 *    Q4_K 144 B / 256 {d, dmin f16, scales[12], qs[128]}; Q5_K 176 B / 256
 *    {d, dmin, scales[12], qh[32], qs[128]}; for both w = d*sc_j*q - dmin*m_j
 *    (OpenVINO PR #38696 "Details"); Q6_K 210 B / 256 {ql[128], qh[64],
 *    scales[16] i8, d f16}, w = d*scales[j]*(q6 - 32).
 *  - Alignment: w, x, y, residual and workspace must be 16-byte aligned.
 *  - All entry points are thread-safe with respect to the host; calls that
 *    share a workspace must be ordered on one stream.
 *
 * Status codes: 0 = OK, negative = error (see gguf_status).  Argument errors
 * are detected on the host before anything is launched.
 */
#ifndef GGUF_MM_H
#define GGUF_MM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* gguf_stream_t; /* same type as cudaStream_t */

/* GGUF type ids.  Q4_0 / Q4_1 / Q5_0 / Q5_1 / Q8_0 hold 32 values per block,
 * the K-quants 256 (GGUF Support Proposal for mobius, 1.2 "Quantization
 * Types"). */
typedef enum {
    GGUF_Q4_0 = 2, GGUF_Q4_1 = 3, GGUF_Q5_0 = 6, GGUF_Q5_1 = 7,
    GGUF_Q8_0 = 8, GGUF_Q2_K = 10, GGUF_Q3_K = 11, GGUF_Q4_K = 12, GGUF_Q5_K = 13, GGUF_Q6_K = 14
} gguf_qtype;

/* GGUF_LAYOUT_Q6K_PLANES: the Q6_K tensor regrouped once into
 * QL[nblk][128] | QH[nblk][64] | SC[nblk][16] | D[nblk] (2 bytes each), same
 * size and contents as the blocks (OpenVINO PR #39119, "Transformation"). */
typedef enum { GGUF_LAYOUT_BLOCKS = 0, GGUF_LAYOUT_Q6K_PLANES = 1 } gguf_layout;

typedef enum { GGUF_DT_F32 = 0, GGUF_DT_F16 = 1, GGUF_DT_BF16 = 2 } gguf_dtype;

/* Execution path of gguf_mm_gemm (OpenVINO PR #39119, "Implementation": the
 * path follows the activation row count; an internal option forces a path).
 * AUTO: fewer activation rows than the format's measured crossover (see
 * gguf_mm_auto_path), or f32 activations with at most 8 rows -> GEMV;
 * otherwise the fused tensor-core GEMM. */
typedef enum { GGUF_PATH_AUTO = 0, GGUF_PATH_GEMV = 1, GGUF_PATH_FUSED = 2 } gguf_path;

typedef enum {
    GGUF_OK = 0,
    GGUF_ERR_INVALID_ARG = -1,  /* null pointer, non-positive size, K not a multiple of the block */
    GGUF_ERR_UNSUPPORTED = -2,  /* type / layout / dtype / size combination not implemented */
    GGUF_ERR_MISALIGNED = -3,   /* a pointer is not 16-byte aligned */
    GGUF_ERR_WORKSPACE = -4,    /* workspace missing or smaller than gguf_mm_workspace_size() */
    GGUF_ERR_CUDA = -5,         /* a CUDA runtime call or kernel launch failed */
    GGUF_ERR_TIMEOUT = -6,      /* a bounded device-side wait expired (reported by check_errors) */
    GGUF_ERR_NO_DEVICE = -7,    /* no sm_103 device current */
    GGUF_ERR_IO = -8,           /* gguf_file_*: the file cannot be opened, read or mapped */
    GGUF_ERR_FORMAT = -9,       /* gguf_file_*: not a GGUF v2/v3 file, or a field runs past its end */
    GGUF_ERR_NOT_FOUND = -10    /* gguf_file_*: no tensor or key of that name */
} gguf_status;

typedef enum { GGUF_OP_GEMV = 0, GGUF_OP_GEMM = 1, GGUF_OP_ID = 2, GGUF_OP_DENSE = 3 } gguf_op;

/* Bytes of device workspace the given call needs (0 = none; pass NULL then).
 * op GGUF_OP_GEMV/GEMM take (t, N, K, M) -- the GEMM figure also covers the
 * GEMV path that GGUF_PATH_AUTO/GEMV may take for M <= 8; GGUF_OP_ID takes all arguments with M
 * the token count T; GGUF_OP_DENSE takes (N, K, M).  Returns 0 for invalid input.
 * The GGUF_OP_GEMM figure depends on the current device's SM count (152 is
 * assumed when no device is current): query it on the device that runs the
 * call. */
size_t gguf_mm_workspace_size(int op, int qtype, int64_t N, int64_t K, int64_t M,
                              int64_t n_expert, int64_t top_k);

/* Decode GEMV: Y[m, n] = sum_k X[m, k] * W[n, k] (+ residual[m, n]) for M <= 8.
 * (OpenVINO PR #39119, "Implementation", GEMV row: activations are quantized per
 * 32 values to int8 with one f32 scale per block -- d_a = amax/127, q =
 * round(x/d_a) -- and every weight sub-block is dotted in integers against them.)
 *   w        [N, K/blk*bb] u8 blocks, or Q6_K planes when layout = PLANES
 *   qtype    any of the ten GGUF_Q* formats;  K a multiple of the format's
 *            block (256 values for the K-quants, 32 for the others)
 *   x        [M, K] of xdt (F32, F16 or BF16), 1 <= M <= 8
 *   residual [M, N] of ydt or NULL;  y [M, N] of ydt
 *   workspace  device buffer of at least gguf_mm_workspace_size(GGUF_OP_GEMV,
 *              qtype, N, K, M, 0, 0) bytes, caller-owned, 16-byte aligned.  On
 *              the paths with a separate quantizer kernel, that kernel writes
 *              the quantized activations there (codes, then per-32 {d_a,
 *              d_a*s, s_lo, s_hi}) and the GEMV kernel copies that image into
 *              every CTA's shared memory.  Its contents are meaningless between
 *              calls.
 * Q4_K / Q5_K at M <= 4 run one kernel that quantizes X itself; from M = 2
 * on its CTAs run in clusters of two that share that quantization through
 * distributed shared memory (GGUF_MM_GEMV_CLUSTER = 1, 2 or 4 in the
 * environment, read at each call, sets the cluster size for comparison runs;
 * the results are the same).
 * Errors: INVALID_ARG, UNSUPPORTED (M > 8, M*K too large for on-chip staging),
 * WORKSPACE (missing or too small), MISALIGNED, CUDA.
 * Weights are static inputs: the kernel is launched with programmatic
 * dependent launch and starts fetching w while the kernel before it on the
 * stream may still be running (x and residual are read, and y written, only
 * after that kernel has finished).  So w must be complete before the preceding
 * kernel on the stream starts; a weight written by a kernel right before this
 * call needs a stream/event synchronization in between, or GGUF_MM_PDL=0 in the
 * environment, which turns the early fetch off.  The workspace is written only
 * after the preceding kernel has finished. */
int gguf_mm_gemv(const void* w, int qtype, int layout, int64_t N, int64_t K,
                 const void* x, int xdt, int64_t M, const void* residual, void* y, int ydt,
                 void* workspace, size_t ws_bytes, gguf_stream_t stream);

/* gguf_mm_gemv from host memory, end to end, in one call: enqueues on `stream`
 * the copy of x_host (and residual_host) into the caller's device buffers
 * x_dev (residual_dev), the GEMV of gguf_mm_gemv on them into y_dev, and the
 * copy of y_dev back into y_host.  Asynchronous: the host buffers must stay
 * valid, and y_host unread, until the stream has passed the call (pinned host
 * memory lets the copies run asynchronously; pageable memory makes the
 * runtime stage them).
 *   x_host, x_dev              [M, K] of xdt (host / device)
 *   residual_host, residual_dev  [M, N] of ydt, both NULL or both set (the
 *                              device one may alias y_dev)
 *   y_host, y_dev              [M, N] of ydt (host / device)
 *   the other arguments as gguf_mm_gemv (w and workspace in device memory).
 * Errors: INVALID_ARG (a missing host buffer, or only one of the residual
 * pair), then those of gguf_mm_gemv, all returned before anything is
 * enqueued; CUDA for a copy the runtime refused. */
int gguf_mm_gemv_host(const void* w, int qtype, int layout, int64_t N, int64_t K,
                      const void* x_host, void* x_dev, int xdt, int64_t M,
                      const void* residual_host, void* residual_dev,
                      void* y_host, void* y_dev, int ydt,
                      void* workspace, size_t ws_bytes, gguf_stream_t stream);

/* The path GGUF_PATH_AUTO takes for this call shape (GGUF_PATH_GEMV or
 * GGUF_PATH_FUSED), or GGUF_ERR_INVALID_ARG.  The GEMV takes M below the
 * smallest row count at which the fused GEMM measured faster on GB300 for the
 * format and shape class (at most 8192 weight rows, or more): Q4_K 9 / 7,
 * Q5_K 9 / 6, Q6_K planes 8 / 5, raw Q6_K 4 / 3, Q8_0 6 / 2; other formats 8
 * (the pages' threshold).  f32 activations stay on the GEMV up to 8 rows. */
int gguf_mm_auto_path(int qtype, int layout, int64_t N, int64_t K, int64_t M, int xdt);

/* Prefill GEMM (or GEMV when the path says so), same arguments and semantics as
 * gguf_mm_gemv plus `path` (gguf_path) and any M >= 1.  The fused path stages
 * weight blocks in shared memory, decodes each 256-value block once to f16 and
 * feeds it to tcgen05 tensor-core MMAs with TMEM accumulators; activations are
 * converted to f16 into the workspace first (OpenVINO PR #39119,
 * "Implementation", DPAS prefill row: decode each block once, reuse it across
 * activation rows, overlap loading with decoding, tile grows with M).  When
 * the weight's row tiles are too few to occupy the GPU (small N), K is split
 * across CTAs: each slice's partial sums go to the workspace and the last
 * slice to finish a tile adds them in slice order (the result does not depend
 * on timing).
 * Workspace: gguf_mm_workspace_size(GGUF_OP_GEMM, ...) bytes. */
int gguf_mm_gemm(const void* w, int qtype, int layout, int64_t N, int64_t K,
                 const void* x, int xdt, int64_t M, const void* residual, void* y, int ydt,
                 void* workspace, size_t ws_bytes, int path, gguf_stream_t stream);

/* MoE expert GEMM (llama.cpp PR #28301 "metal : skip the empty half of the
 * mul_mm_id token tile", "Overview"): for every token t and slot k,
 *   Y[t, k, :] = X[t, :] . W_{ids[t, k]}^T (+ residual[t, k, :]).
 *   w_experts n_expert weight tensors [N, K/blk*bb] back to back (Q4_K/Q5_K/Q6_K/Q8_0 blocks)
 *   x [T, K] of xdt (F16 or BF16); ids [T, top_k] int32 (device), each in [0, n_expert)
 *   residual [T, top_k, N] of ydt or NULL;  y [T, top_k, N] of ydt (F32, F16, BF16)
 * Rows are grouped by expert on the device; each (expert, 128-row weight tile,
 * token tile) issues MMAs only for round_up(rows, 16) token columns, so the
 * empty part of an underfilled token tile costs nothing.  (For comparison
 * runs, the environment variable GGUF_MM_MOE_FULL_TILES=1, read at each call,
 * issues every tile's MMAs at the full width instead; the output is the same.)
 * Ids outside [0, n_expert) are skipped (their Y rows are left untouched).
 * Decode form (mul_mv_id): when T * top_k is at most 128 (Q4_K, Q5_K, Q2_K,
 * Q3_K, Q6_K experts), 32 (Q4_0, Q4_1, Q5_0, Q5_1) or 16 (Q8_0), every routed
 * row is instead one GEMV of the decode path (int8 activation codes, integer
 * sub-block dots; the results are those of gguf_mm_gemv on that expert and
 * row), with no routing step.
 * GGUF_MM_MOE_MV=0 in the environment keeps every batch on the routed path.
 * Workspace: gguf_mm_workspace_size(GGUF_OP_ID, ...) bytes. */
int gguf_mm_id(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K,
               const void* x, int xdt, int64_t T, const int32_t* ids, int64_t top_k,
               const void* residual, void* y, int ydt,
               void* workspace, size_t ws_bytes, gguf_stream_t stream);

/* The same expert GEMM with one activation row per (token, slot) -- the
 * down-projection form of mul_mm_id, where each slot's input is that
 * expert's own up-projection output (llama.cpp PR #28301, "Overview": every
 * routed row multiplies its expert's weight):
 *   Y[t, k, :] = X[t, k, :] . W_{ids[t, k]}^T (+ residual[t, k, :]),
 *   x [T, top_k, K] of xdt (F16 or BF16); all other arguments, the workspace
 *   size (gguf_mm_workspace_size(GGUF_OP_ID, ...)) and the errors as gguf_mm_id. */
int gguf_mm_id_slots(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K,
                     const void* x, int xdt, int64_t T, const int32_t* ids, int64_t top_k,
                     const void* residual, void* y, int ydt,
                     void* workspace, size_t ws_bytes, gguf_stream_t stream);

/* The form gguf_mm_id / gguf_mm_id_slots take for T tokens of top_k routed
 * rows of qtype experts: GGUF_PATH_GEMV (the decode form) or GGUF_PATH_FUSED
 * (the routed tensor-core path); GGUF_ERR_INVALID_ARG for a bad argument.
 * Host only: nothing is launched and no GPU is needed. */
int gguf_mm_id_form(int qtype, int64_t T, int64_t top_k);

/* gguf_mm_id (per_slot = 0) or gguf_mm_id_slots (per_slot = 1) with the form
 * chosen by the caller instead of by the batch size:
 *   path = GGUF_PATH_AUTO   the batch-size rule of gguf_mm_id;
 *          GGUF_PATH_GEMV   the decode form (int8 activation codes, the
 *                           GEMV's arithmetic) for any format, at most 128
 *                           routed rows (T * top_k), else UNSUPPORTED;
 *          GGUF_PATH_FUSED  the routed tensor-core path (f16 operands, f32
 *                           accumulation) at every batch size.
 * So a caller that needs one arithmetic for every batch size can fix it.
 * All other arguments, the workspace size and the errors as gguf_mm_id;
 * INVALID_ARG for another path value. */
int gguf_mm_id_path(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K,
                    const void* x, int xdt, int64_t T, const int32_t* ids, int64_t top_k, int per_slot,
                    const void* residual, void* y, int ydt,
                    void* workspace, size_t ws_bytes, int path, gguf_stream_t stream);

/* Q6_K plane regrouping (OpenVINO PR #39119, "Transformation"): blocks ->
 * QL[nblk][128] | QH[nblk][64] | SC[nblk][16] | D[nblk][2] (inverse = 0), or
 * back (inverse = 1).  src and dst are 210*nblk bytes each and must not
 * overlap; blocks are in row-major (n, kb) order.  Done once per weight. */
int gguf_repack_q6k_planes(const void* src, void* dst, int64_t nblk, int inverse,
                           gguf_stream_t stream);

/* Decode-once to a K-padded buffer (ROCm llama.cpp PR #37 "one-time K-padded
 * f16 dequantization for prefill GEMMs", "How it works"): out[n, k] = w[n, k]
 * rounded to odt (F16 or BF16) for k < K and 0 for K <= k < ld.  ld >= K, ld % 8
 * == 0; ld = K + 64 pads each row by one 128-byte line. */
int gguf_dequant_padded(const void* w, int qtype, int layout, int64_t N, int64_t K,
                        void* out, int odt, int64_t ld, gguf_stream_t stream);

/* Dense tensor-core GEMM on a decoded weight: Y[m, n] = sum_k X[m, k] * Wd[n, k]
 * (+ residual), Wd [N, ld] of wdt (F16 or BF16), X [M, K] of xdt (F16/BF16);
 * activations are converted to wdt into the workspace first
 * (gguf_mm_workspace_size(GGUF_OP_DENSE, 0, N, K, M, 0, 0) bytes).
 * K % 64 == 0, ld % 8 == 0. */
int gguf_dense_gemm(const void* wdense, int wdt, int64_t ld, int64_t N, int64_t K,
                    const void* x, int xdt, int64_t M, const void* residual, void* y, int ydt,
                    void* workspace, size_t ws_bytes, gguf_stream_t stream);

/* Allocation-free form of gguf_dense_gemm, for callers that may not obtain
 * device memory (their host program owns every allocation, or a cudaMalloc
 * there would synchronize the device at the wrong moment): same arguments
 * minus the workspace; the scratch this call needs (the activations converted
 * to wdt, M*K*2 bytes) lives in an 8 MiB array built into the library, which
 * every GPU that loads the library keeps until the process exits.  The pages
 * have no counterpart of this entry point.
 *   - M*K*2 > 8 MiB returns GGUF_ERR_WORKSPACE before anything is launched.
 *   - The call allocates nothing.  Its first call on a device looks up the
 *     array's device address (cudaGetSymbolAddress, with that device current);
 *     make that first call before any stream capture.
 *   - All calls share the one array and each overwrites, before reading, the
 *     part it uses, so nothing in it needs to start at zero; calls that overlap
 *     on the GPU (other streams, other host threads) race on it. */
int gguf_dense_gemm_noalloc(const void* wdense, int wdt, int64_t ld, int64_t N, int64_t K,
                            const void* x, int xdt, int64_t M, const void* residual, void* y, int ydt,
                            gguf_stream_t stream);

/* Synchronises `stream`, then returns and clears the device status word of the
 * current device: GGUF_OK, GGUF_ERR_TIMEOUT (a bounded wait in a kernel expired;
 * that kernel's outputs are undefined), or GGUF_ERR_CUDA for a pending CUDA error. */
int gguf_mm_check_errors(gguf_stream_t stream);

/* Static string for a status code. */
const char* gguf_mm_status_string(int status);

/* Library ABI version (major*100 + minor). */
int gguf_mm_version(void);

/* Test hook: runs gguf_mm_gemv (same arguments and workspace rules) with a
 * build of its GEMV kernel that also writes the integer intermediates, so they
 * can be compared bit for bit with a CPU restatement: qa [M, K] i8, d_a
 * [M, K/32] f32 and s [M, K/32] i32 from the activation quantizer (taken from
 * the first CTA), and the integer sub-block dots D [M, N, K/sub] i32, sub = 16
 * for Q6_K and 32 otherwise.  Q6_K dots are of (q6 - 32), Q4_K/Q5_K of the
 * unsigned quant, Q8_0 of the signed quant.  Any debug pointer may be NULL.
 *   kernel      -1: the kernel gguf_mm_gemv would choose; else one of the
 *               GEMV kernel ids below, forced (UNSUPPORTED if it cannot run
 *               this shape)
 *   kernel_out  host int* or NULL: receives the id of the kernel that ran
 * Kernel ids: 0 staged rows (per-warp ring of row slots), 1 direct register
 * loads, 2 tile (M = 1, whole rows in shared memory, quantizer inside), 3 pair
 * (M = 2..4, activation codes in registers), 4 row-lane (M = 1..4, a lane per
 * weight row, quantizer inside).  Allocates nothing. */
int gguf_mm_debug_gemv_terms(const void* w, int qtype, int layout, int64_t N, int64_t K,
                             const void* x, int xdt, int64_t M, const void* residual, void* y, int ydt,
                             int8_t* qa, float* d_a, int32_t* s, int32_t* D,
                             void* workspace, size_t ws_bytes, int kernel, int* kernel_out,
                             gguf_stream_t stream);

/* The GEMV kernel id (as above) that gguf_mm_gemv chooses for this shape on the
 * current device, or a negative status.  Launches nothing. */
int gguf_mm_gemv_kernel(int qtype, int layout, int64_t N, int64_t K, int64_t M, int xdt);

/* Test hook: the MoE routing step of gguf_mm_id alone, writing its tables
 * into caller buffers (device memory) so that they can be compared with a CPU
 * restatement: for ids [entries] int32 (entries = T * top_k; ids outside
 * [0, n_expert) are skipped),
 *   offsets [n_expert + 1]  start of each expert's group of rows; offsets[E]
 *                           = number of routed rows (integer, exact)
 *   ntiles  [1]             number of (expert, token tile of <= 128 rows) items
 *   tiles   [max_tiles][4]  the items {expert, first row in the group, rows, 0}
 *   rows    [entries]       the routed entries (token * top_k + slot), grouped
 *                           by expert; the order inside a group is unspecified
 * max_tiles must be at least min(n_expert, entries) + ceil(entries / 128)
 * (else WORKSPACE); tiles must be 16-byte aligned. */
int gguf_mm_debug_moe_route(const int32_t* ids, int64_t entries, int64_t n_expert, int32_t* offsets,
                            int32_t* ntiles, int32_t* tiles, int64_t max_tiles, int32_t* rows,
                            gguf_stream_t stream);

/* Test hook: gguf_mm_id (per_slot = 0) or gguf_mm_id_slots (per_slot = 1) in
 * its decode form for Q4_K / Q5_K experts (at most 128 routed rows; other
 * formats and larger batches give GGUF_ERR_UNSUPPORTED) --
 * with the integer intermediates of every routed row p = token * top_k + slot
 * whose expert id is valid written out (device memory; any may be NULL):
 *   qa [entries, K] int8, d_a [entries, K/32] f32, s [entries, K/32] int32
 *   (the row's activation codes, scales and code sums, as gguf_mm_debug_gemv_terms)
 *   D  [entries, N, K/32] int32 (the sub-block dots of row p against its expert)
 * Rows with an invalid id are left untouched.  Allocates nothing. */
int gguf_mm_debug_moe_mv_terms(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K,
                               const void* x, int xdt, int64_t T, const int32_t* ids, int64_t top_k, int per_slot,
                               const void* residual, void* y, int ydt, int8_t* qa, float* d_a, int32_t* s,
                               int32_t* D, void* workspace, size_t ws_bytes, gguf_stream_t stream);

/* Test hook for the bounded device waits: launches a kernel whose wait on an
 * mbarrier that nothing completes gives up after about `spin_limit` polls and
 * records GGUF_ERR_TIMEOUT in the device status word (read it with
 * gguf_mm_check_errors).  No GPU fault is involved. */
int gguf_mm_debug_timeout(int64_t spin_limit, gguf_stream_t stream);

/* ---------------------------------------------------------------------------
 * GGUF container reader (host only: no device memory, no CUDA call)
 *
 * A .gguf file holds the model's metadata as key-value pairs and its tensors,
 * each with its own type (GGUF Support Proposal for mobius, 1.1 "Overview";
 * the tensor names of 1.3).  The reader memory-maps the file, parses the
 * header, the key-value pairs and the tensor table, and checks every field
 * against the file's size: a truncated or malformed file gives
 * GGUF_ERR_FORMAT, never a read past the mapping.  Versions 2 and 3 of the
 * published container layout are read (little-endian):
 *   "GGUF" u32 version, u64 n_tensors, u64 n_kv, n_kv x {string key, u32
 *   value type, value}, n_tensors x {string name, u32 n_dims, u64 dims[],
 *   u32 type, u64 offset}, padding to general.alignment (default 32), data.
 * Value types: 0 u8, 1 i8, 2 u16, 3 i16, 4 u32, 5 i32, 6 f32, 7 bool,
 * 8 string, 9 array, 10 u64, 11 i64, 12 f64.  Tensor dims[0] is the
 * contiguous dimension: a weight W[N, K] has dims {K, N}, and its bytes are
 * exactly the [N, K/blk*bb] block array the matmul entry points take.
 * A handle is used by one thread at a time; distinct handles are independent.
 * ------------------------------------------------------------------------- */
typedef struct gguf_file* gguf_file_t;

/* Opens and parses `path`; *out receives the handle (NULL on error).
 * GGUF_ERR_IO (open/stat/mmap failed), GGUF_ERR_FORMAT. */
int gguf_file_open(const char* path, gguf_file_t* out);
void gguf_file_close(gguf_file_t f);              /* NULL is a no-op */
int gguf_file_version(gguf_file_t f);             /* 2 or 3 */
int64_t gguf_file_alignment(gguf_file_t f);       /* data alignment in bytes */
int64_t gguf_file_tensor_count(gguf_file_t f);

/* Tensor `index`: its name (NUL-terminated into name[name_cap], WORKSPACE when
 * it does not fit), GGUF type id, number of dims, dims (unused ones 1), the
 * absolute file offset of its data and its size in bytes (0 when the type's
 * size is not known to the reader: known are F32 0, F16 1, BF16 30, Q4_0,
 * Q4_1, Q5_0, Q5_1, Q8_0, Q2_K 10, Q3_K 11, Q4_K, Q5_K, Q6_K).  Any output
 * pointer may be NULL. */
int gguf_file_tensor_info(gguf_file_t f, int64_t index, char* name, size_t name_cap, int* type, int* n_dims,
                          int64_t dims[4], uint64_t* file_offset, uint64_t* nbytes);

/* Index of the tensor called `name`, or GGUF_ERR_NOT_FOUND. */
int64_t gguf_file_find_tensor(gguf_file_t f, const char* name);

/* Copies tensor `index`'s bytes into HOST memory host_dst[dst_bytes]
 * (WORKSPACE when smaller than the tensor, UNSUPPORTED when its size is
 * unknown).  Copy them to the device with one cudaMemcpy to run a matmul. */
int gguf_file_read_tensor(gguf_file_t f, int64_t index, void* host_dst, size_t dst_bytes);

/* For a 2-D tensor of a type the matmul entry points take (gguf_qtype):
 * its qtype, N = dims[1] and K = dims[0].  UNSUPPORTED otherwise. */
int gguf_file_tensor_as_weight(gguf_file_t f, int64_t index, int* qtype, int64_t* N, int64_t* K);

int64_t gguf_file_kv_count(gguf_file_t f);
/* Key of pair `index` into key[cap] and its value type (either may be NULL). */
int gguf_file_kv_key(gguf_file_t f, int64_t index, char* key, size_t cap, int* value_type);
/* Value of `key` as an integer (any integer or bool type; a u64 above
 * INT64_MAX is UNSUPPORTED) or a float (f32, f64 or any integer type).
 * NOT_FOUND, UNSUPPORTED for another value type. */
int gguf_file_get_int(gguf_file_t f, const char* key, int64_t* out);
int gguf_file_get_float(gguf_file_t f, const char* key, double* out);
/* A string value: *len receives its byte length; buf (may be NULL) receives
 * the bytes plus a NUL when cap > len (else WORKSPACE). */
int gguf_file_get_string(gguf_file_t f, const char* key, char* buf, size_t cap, size_t* len);
/* An array value: its element type and count; dst (may be NULL) receives the
 * elements of a scalar array (cap bytes; WORKSPACE when smaller).  String
 * arrays report type and count only. */
int gguf_file_get_array(gguf_file_t f, const char* key, int* elem_type, int64_t* count, void* dst, size_t cap);

#ifdef __cplusplus
}
#endif

#endif /* GGUF_MM_H */
