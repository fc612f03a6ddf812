// C ABI of libgguf_mm.so: argument validation, per-device launch facts, the
// device status word, and dispatch to the kernels.  Nothing here allocates
// device memory: every buffer is the caller's, and the status word is a
// module-scope __device__ variable.
#include <algorithm>
#include <mutex>
#include <cstring>
#include <cstdlib>

#include "common.cuh"
#include "formats.cuh"
#include "gemv.cuh"
#include "gemm.cuh"
#include "moe.cuh"

namespace gg {
cudaError_t repack_q6k_launch(const void* src, void* dst, int64_t nblk, int inverse, cudaStream_t stream);
cudaError_t dequant_padded_launch(const void* w, int qtype, int layout, int64_t N, int64_t K, void* out, int odt,
                                  int64_t ld, int num_sms, cudaStream_t s);
}  // namespace gg

using namespace gg;

// One status word per device: the first failing bounded wait writes its code.
__device__ int g_status_word;

namespace {

struct DeviceFacts {
    bool ready = false;
    int num_sms = 0;
    int max_smem_optin = 0;
    int cc_major = 0, cc_minor = 0;
    int* status = nullptr;  // device address of g_status_word
};

constexpr int kMaxDevices = 64;
DeviceFacts g_facts[kMaxDevices];
std::mutex g_facts_mu;

int facts(DeviceFacts** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GGUF_ERR_NO_DEVICE;
    std::lock_guard<std::mutex> lk(g_facts_mu);
    DeviceFacts& f = g_facts[dev];
    if (!f.ready) {
        if (cudaDeviceGetAttribute(&f.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&f.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&f.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&f.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
            return GGUF_ERR_CUDA;
        // the kernels are built for sm_103a only
        if (f.cc_major != 10 || f.cc_minor != 3) return GGUF_ERR_NO_DEVICE;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return GGUF_ERR_CUDA;
        f.status = static_cast<int*>(p);
        f.ready = true;
    }
    *out = &f;
    return GGUF_OK;
}

// Programmatic dependent launch for the GEMV (on unless GGUF_MM_PDL=0).
bool pdl_enabled() {
    static const bool on = [] {
        const char* e = getenv("GGUF_MM_PDL");
        return !(e && e[0] == '0');
    }();
    return on;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool valid_qtype(int t) {
    return t == GGUF_Q4_0 || t == GGUF_Q4_1 || t == GGUF_Q5_0 || t == GGUF_Q5_1 || t == GGUF_Q8_0 || t == GGUF_Q2_K ||
           t == GGUF_Q3_K || t == GGUF_Q4_K || t == GGUF_Q5_K || t == GGUF_Q6_K;
}
bool valid_dtype(int d) { return d == GGUF_DT_F32 || d == GGUF_DT_F16 || d == GGUF_DT_BF16; }

// Shared checks of the weight / shape / pointer arguments.
int check_common(const void* w, int qtype, int layout, int64_t N, int64_t K, const void* x, int xdt, int64_t M,
                 const void* residual, const void* y, int ydt) {
    if (!w || !x || !y) return GGUF_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || M <= 0) return GGUF_ERR_INVALID_ARG;
    if (!valid_qtype(qtype) || !valid_dtype(xdt) || !valid_dtype(ydt)) return GGUF_ERR_UNSUPPORTED;
    if (K % block_values(qtype) != 0) return GGUF_ERR_INVALID_ARG;
    if (layout != GGUF_LAYOUT_BLOCKS && layout != GGUF_LAYOUT_Q6K_PLANES) return GGUF_ERR_UNSUPPORTED;
    if (layout == GGUF_LAYOUT_Q6K_PLANES && qtype != GGUF_Q6_K) return GGUF_ERR_UNSUPPORTED;
    if (!aligned16(w) || !aligned16(x) || !aligned16(y) || (residual && !aligned16(residual)))
        return GGUF_ERR_MISALIGNED;
    if (N > (int64_t(1) << 31) || K > (int64_t(1) << 24) || M > (int64_t(1) << 24)) return GGUF_ERR_UNSUPPORTED;
    return GGUF_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? GGUF_OK : GGUF_ERR_CUDA; }

// The smallest activation row count at which the fused GEMM beat the GEMV on
// GB300, per format and shape class (chains of calls on weight copies larger
// than L2, bf16 activations; the crossover table of bench.py --crossover):
// at most 8192 weight rows (measured at 4096 x 4096: at most 64 tiles of 128
// rows for 152 SMs, so the fused path splits K) and more (14336 x 4096).  A
// value above 8 keeps every row count the GEMV can take on the GEMV.
int crossover_rows(int qtype, int layout, int64_t N, int64_t K) {
    (void)K;
    const bool large = N > 8192;
    switch (qtype) {
        case GGUF_Q4_K: return large ? 7 : 9;
        case GGUF_Q5_K: return large ? 6 : 9;
        case GGUF_Q6_K:
            return layout == GGUF_LAYOUT_Q6K_PLANES ? (large ? 4 : 7) : (large ? 2 : 3);
        case GGUF_Q8_0: return large ? 2 : 6;
        case GGUF_Q4_0: return large ? 2 : 6;
        case GGUF_Q4_1: return large ? 3 : 6;
        case GGUF_Q5_0: return large ? 3 : 6;
        case GGUF_Q5_1: return large ? 2 : 5;
        case GGUF_Q2_K: return large ? 2 : 4;
        case GGUF_Q3_K: return large ? 4 : 5;
        default: return 8;
    }
}

// GGUF_PATH_AUTO's choice.  OpenVINO PR #39119, "Implementation", path table:
// few activation rows or f32 activations -> GEMV, otherwise the prefill GEMM;
// "few" is the measured crossover above (the pages' Xe threshold is 8), and
// f32 activations stay on the GEMV up to the 8 rows it takes.
int auto_path(int qtype, int layout, int64_t N, int64_t K, int64_t M, int xdt) {
    if (M <= 8 && M < crossover_rows(qtype, layout, N, K)) return GGUF_PATH_GEMV;
    if (xdt == GGUF_DT_F32 && M <= 8) return GGUF_PATH_GEMV;
    return GGUF_PATH_FUSED;
}

int run_gemv(const void* w, int qtype, int layout, int64_t N, int64_t K, const void* x, int xdt, int64_t M,
             const void* residual, void* y, int ydt, void* workspace, size_t ws_bytes, cudaStream_t stream,
             int8_t* qa, float* da, int32_t* s, int32_t* D, bool dump, int force = -1, int* kind = nullptr,
             bool launch = true) {
    int st = check_common(w, qtype, layout, N, K, x, xdt, M, residual, y, ydt);
    if (st != GGUF_OK) return st;
    if (M > 8) return GGUF_ERR_UNSUPPORTED;
    if (!workspace || ws_bytes < gemv_workspace_bytes(M, K)) return GGUF_ERR_WORKSPACE;
    if (!aligned16(workspace)) return GGUF_ERR_MISALIGNED;
    DeviceFacts* f = nullptr;
    if ((st = facts(&f)) != GGUF_OK) return st;
    GemvParams p{};
    p.w = static_cast<const uint8_t*>(w);
    p.qtype = qtype;
    p.layout = layout;
    p.N = N;
    p.K = K;
    p.x = x;
    p.xdt = xdt;
    p.M = (int)M;
    p.residual = residual;
    p.y = y;
    p.ydt = ydt;
    p.status = f->status;
    p.pdl = pdl_enabled() ? 1 : 0;
    p.act_image = workspace;
    p.dbg_qa = qa;
    p.dbg_da = da;
    p.dbg_s = s;
    p.dbg_D = D;
    p.force = force;
    int grid = 0;
    size_t smem = 0;
    if ((st = gemv_plan(p, f->num_sms, f->max_smem_optin, &grid, &smem)) != GGUF_OK) return st;
    if (kind) *kind = gemv_kind(p);
    if (!launch) return GGUF_OK;
    return cuda_status(gemv_launch(p, grid, smem, dump, stream));
}

__global__ void timeout_probe_kernel(long long limit, int* status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // nothing ever arrives on `bar`: the bounded wait must give up and report
    if (threadIdx.x == 0) mbar_wait(&bar, 0, status, limit);
}

}  // namespace

int gg::current_device_launch_facts(int* num_sms, int** status) {
    DeviceFacts* f = nullptr;
    const int st = facts(&f);
    if (st != GGUF_OK) return st;
    *num_sms = f->num_sms;
    *status = f->status;
    return GGUF_OK;
}

extern "C" {

int gguf_mm_version(void) { return 100; }

const char* gguf_mm_status_string(int status) {
    switch (status) {
        case GGUF_OK: return "ok";
        case GGUF_ERR_INVALID_ARG: return "invalid argument";
        case GGUF_ERR_UNSUPPORTED: return "unsupported type/layout/dtype/size combination";
        case GGUF_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case GGUF_ERR_WORKSPACE: return "workspace missing or too small";
        case GGUF_ERR_CUDA: return "CUDA error";
        case GGUF_ERR_TIMEOUT: return "bounded device wait expired";
        case GGUF_ERR_NO_DEVICE: return "no sm_103 device current";
        case GGUF_ERR_IO: return "file cannot be opened or mapped";
        case GGUF_ERR_FORMAT: return "not a well-formed GGUF v2/v3 file";
        case GGUF_ERR_NOT_FOUND: return "no tensor or key of that name";
        default: return "unknown status";
    }
}

size_t gguf_mm_workspace_size(int op, int qtype, int64_t N, int64_t K, int64_t M, int64_t n_expert,
                              int64_t top_k) {
    if (N <= 0 || K <= 0 || M <= 0) return 0;
    switch (op) {
        case GGUF_OP_GEMV: return M <= 8 ? gemv_workspace_bytes(M, K) : 0;
        case GGUF_OP_GEMM: {
            // sized for the current device's SM count (152 when none is current)
            int sms = 152, *st = nullptr;
            if (gg::current_device_launch_facts(&sms, &st) != GGUF_OK) sms = 152;
            return std::max(gemm_workspace_bytes(qtype, N, K, M, sms), M <= 8 ? gemv_workspace_bytes(M, K) : size_t(0));
        }
        case GGUF_OP_DENSE: return dense_workspace_bytes(N, K, M);
        case GGUF_OP_ID:
            if (n_expert <= 0 || top_k <= 0) return 0;
            return moe_workspace_bytes(qtype, n_expert, N, K, M, top_k);
        default: return 0;
    }
}

int gguf_mm_gemv(const void* w, int qtype, int layout, int64_t N, int64_t K, const void* x, int xdt, int64_t M,
                 const void* residual, void* y, int ydt, void* workspace, size_t ws_bytes,
                 gguf_stream_t stream) {
    return run_gemv(w, qtype, layout, N, K, x, xdt, M, residual, y, ydt, workspace, ws_bytes, (cudaStream_t)stream,
                    nullptr, nullptr, nullptr, nullptr, false);
}

int gguf_mm_gemv_host(const void* w, int qtype, int layout, int64_t N, int64_t K, const void* x_host, void* x_dev,
                      int xdt, int64_t M, const void* residual_host, void* residual_dev, void* y_host, void* y_dev,
                      int ydt, void* workspace, size_t ws_bytes, gguf_stream_t stream) {
    if (!x_host || !y_host || (residual_host == nullptr) != (residual_dev == nullptr)) return GGUF_ERR_INVALID_ARG;
    const cudaStream_t s = (cudaStream_t)stream;
    // every argument of the GEMV checked (its plan, nothing launched) before anything is enqueued
    int st = run_gemv(w, qtype, layout, N, K, x_dev, xdt, M, residual_dev, y_dev, ydt, workspace, ws_bytes, s, nullptr,
                      nullptr, nullptr, nullptr, false, -1, nullptr, false);
    if (st != GGUF_OK) return st;
    const size_t xb = (size_t)(M * K) * (xdt == GGUF_DT_F32 ? 4 : 2), yb = (size_t)(M * N) * (ydt == GGUF_DT_F32 ? 4 : 2);
    if (cudaMemcpyAsync(x_dev, x_host, xb, cudaMemcpyHostToDevice, s) != cudaSuccess) return GGUF_ERR_CUDA;
    if (residual_host && cudaMemcpyAsync(residual_dev, residual_host, yb, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return GGUF_ERR_CUDA;
    st = run_gemv(w, qtype, layout, N, K, x_dev, xdt, M, residual_dev, y_dev, ydt, workspace, ws_bytes, s, nullptr,
                  nullptr, nullptr, nullptr, false);
    if (st != GGUF_OK) return st;
    return cuda_status(cudaMemcpyAsync(y_host, y_dev, yb, cudaMemcpyDeviceToHost, s));
}

int gguf_mm_debug_gemv_terms(const void* w, int qtype, int layout, int64_t N, int64_t K, const void* x, int xdt,
                             int64_t M, const void* residual, void* y, int ydt, int8_t* qa, float* d_a, int32_t* s,
                             int32_t* D, void* workspace, size_t ws_bytes, int kernel, int* kernel_out,
                             gguf_stream_t stream) {
    return run_gemv(w, qtype, layout, N, K, x, xdt, M, residual, y, ydt, workspace, ws_bytes, (cudaStream_t)stream,
                    qa, d_a, s, D, true, kernel, kernel_out);
}

int gguf_mm_auto_path(int qtype, int layout, int64_t N, int64_t K, int64_t M, int xdt) {
    if (!valid_qtype(qtype) || !valid_dtype(xdt) || N <= 0 || K <= 0 || M <= 0) return GGUF_ERR_INVALID_ARG;
    return auto_path(qtype, layout, N, K, M, xdt);
}

int gguf_mm_id_form(int qtype, int64_t T, int64_t top_k) {
    if (!valid_qtype(qtype) || T <= 0 || top_k <= 0 || top_k > 64 || T > (int64_t(1) << 24))
        return GGUF_ERR_INVALID_ARG;
    return moe_decode_form(qtype, T * top_k) ? GGUF_PATH_GEMV : GGUF_PATH_FUSED;
}

int gguf_mm_gemv_kernel(int qtype, int layout, int64_t N, int64_t K, int64_t M, int xdt) {
    // the plan for dummy (aligned, non-null) pointers: nothing is launched
    static const uint8_t dummy[16] __attribute__((aligned(16))) = {};
    const void* d = dummy;
    int kind = -1;
    const int st = run_gemv(d, qtype, layout, N, K, d, xdt, M, nullptr, const_cast<void*>(d), GGUF_DT_F32,
                            const_cast<void*>(d), gemv_workspace_bytes(M > 0 && M <= 8 ? M : 1, K > 0 ? K : 32),
                            nullptr, nullptr, nullptr, nullptr, nullptr, false, -1, &kind, false);
    return st == GGUF_OK ? kind : st;
}

int gguf_mm_gemm(const void* w, int qtype, int layout, int64_t N, int64_t K, const void* x, int xdt, int64_t M,
                 const void* residual, void* y, int ydt, void* workspace, size_t ws_bytes, int path,
                 gguf_stream_t stream) {
    int st = check_common(w, qtype, layout, N, K, x, xdt, M, residual, y, ydt);
    if (st != GGUF_OK) return st;
    if (path != GGUF_PATH_AUTO && path != GGUF_PATH_GEMV && path != GGUF_PATH_FUSED) return GGUF_ERR_INVALID_ARG;
    // the pages' path table: fewer than 8 rows, or f32 activations, to the
    // GEMV; the GEMV takes at most 8 rows, so larger f32 batches go to the
    // fused path (which converts them to f16 row by row)
    if (path == GGUF_PATH_AUTO) path = auto_path(qtype, layout, N, K, M, xdt);
    if (path == GGUF_PATH_GEMV)
        return run_gemv(w, qtype, layout, N, K, x, xdt, M, residual, y, ydt, workspace, ws_bytes,
                        (cudaStream_t)stream, nullptr, nullptr, nullptr, nullptr, false);
    DeviceFacts* f = nullptr;
    if ((st = facts(&f)) != GGUF_OK) return st;
    const size_t need = gemm_workspace_bytes(qtype, N, K, M, f->num_sms);
    if (need && (!workspace || ws_bytes < need)) return GGUF_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return GGUF_ERR_MISALIGNED;
    return gemm_fused_run(w, qtype, layout, N, K, x, xdt, M, residual, y, ydt, workspace, f->num_sms, f->status,
                          (cudaStream_t)stream, pdl_enabled() ? 1 : 0);
}

static int run_id(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K, const void* x, int xdt,
                  int64_t T, const int32_t* ids, int64_t top_k, const void* residual, void* y, int ydt,
                  void* workspace, size_t ws_bytes, gguf_stream_t stream, bool per_slot,
                  const MoeMvDump* dump = nullptr, int form = -1) {
    if (!ids || n_expert <= 0 || top_k <= 0) return GGUF_ERR_INVALID_ARG;
    int st = check_common(w_experts, qtype, GGUF_LAYOUT_BLOCKS, N, K, x, xdt, T, residual, y, ydt);
    if (st != GGUF_OK) return st;
    if (xdt == GGUF_DT_F32) return GGUF_ERR_UNSUPPORTED;
    if (n_expert > 4096 || top_k > 64) return GGUF_ERR_UNSUPPORTED;
    const size_t need = moe_workspace_bytes(qtype, n_expert, N, K, T, top_k);
    if (!workspace || ws_bytes < need) return GGUF_ERR_WORKSPACE;
    if (!aligned16(workspace) || (reinterpret_cast<uintptr_t>(ids) & 3u)) return GGUF_ERR_MISALIGNED;
    DeviceFacts* f = nullptr;
    if ((st = facts(&f)) != GGUF_OK) return st;
    return moe_run(w_experts, qtype, n_expert, N, K, x, xdt, T, ids, top_k, residual, y, ydt, workspace,
                   f->num_sms, f->status, (cudaStream_t)stream, per_slot, dump, pdl_enabled() ? 1 : 0, form);
}

int gguf_mm_debug_moe_mv_terms(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K,
                               const void* x, int xdt, int64_t T, const int32_t* ids, int64_t top_k, int per_slot,
                               const void* residual, void* y, int ydt, int8_t* qa, float* d_a, int32_t* s,
                               int32_t* D, void* workspace, size_t ws_bytes, gguf_stream_t stream) {
    const MoeMvDump dump{qa, d_a, s, D};
    return run_id(w_experts, qtype, n_expert, N, K, x, xdt, T, ids, top_k, residual, y, ydt, workspace, ws_bytes,
                  stream, per_slot != 0, &dump);
}

int gguf_mm_id(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K, const void* x, int xdt,
               int64_t T, const int32_t* ids, int64_t top_k, const void* residual, void* y, int ydt,
               void* workspace, size_t ws_bytes, gguf_stream_t stream) {
    return run_id(w_experts, qtype, n_expert, N, K, x, xdt, T, ids, top_k, residual, y, ydt, workspace, ws_bytes,
                  stream, false);
}

int gguf_mm_id_path(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K, const void* x, int xdt,
                    int64_t T, const int32_t* ids, int64_t top_k, int per_slot, const void* residual, void* y, int ydt,
                    void* workspace, size_t ws_bytes, int path, gguf_stream_t stream) {
    int form;
    switch (path) {
        case GGUF_PATH_AUTO: form = -1; break;
        case GGUF_PATH_GEMV: form = 1; break;    // the decode form
        case GGUF_PATH_FUSED: form = 0; break;   // the routed tensor-core path
        default: return GGUF_ERR_INVALID_ARG;
    }
    return run_id(w_experts, qtype, n_expert, N, K, x, xdt, T, ids, top_k, residual, y, ydt, workspace, ws_bytes,
                  stream, per_slot != 0, nullptr, form);
}

int gguf_mm_id_slots(const void* w_experts, int qtype, int64_t n_expert, int64_t N, int64_t K, const void* x,
                     int xdt, int64_t T, const int32_t* ids, int64_t top_k, const void* residual, void* y, int ydt,
                     void* workspace, size_t ws_bytes, gguf_stream_t stream) {
    return run_id(w_experts, qtype, n_expert, N, K, x, xdt, T, ids, top_k, residual, y, ydt, workspace, ws_bytes,
                  stream, true);
}

int gguf_repack_q6k_planes(const void* src, void* dst, int64_t nblk, int inverse, gguf_stream_t stream) {
    if (!src || !dst || nblk <= 0 || (inverse != 0 && inverse != 1)) return GGUF_ERR_INVALID_ARG;
    if (!aligned16(src) || !aligned16(dst)) return GGUF_ERR_MISALIGNED;
    const uintptr_t a = reinterpret_cast<uintptr_t>(src), b = reinterpret_cast<uintptr_t>(dst);
    const uintptr_t bytes = (uintptr_t)(210 * nblk);
    if (a < b + bytes && b < a + bytes) return GGUF_ERR_INVALID_ARG;  // overlapping
    DeviceFacts* f = nullptr;
    int st = facts(&f);
    if (st != GGUF_OK) return st;
    return cuda_status(repack_q6k_launch(src, dst, nblk, inverse, (cudaStream_t)stream));
}

int gguf_dequant_padded(const void* w, int qtype, int layout, int64_t N, int64_t K, void* out, int odt, int64_t ld,
                        gguf_stream_t stream) {
    if (!w || !out || N <= 0 || K <= 0) return GGUF_ERR_INVALID_ARG;
    if (!valid_qtype(qtype) || (odt != GGUF_DT_F16 && odt != GGUF_DT_BF16)) return GGUF_ERR_UNSUPPORTED;
    if (layout != GGUF_LAYOUT_BLOCKS && layout != GGUF_LAYOUT_Q6K_PLANES) return GGUF_ERR_UNSUPPORTED;
    if (layout == GGUF_LAYOUT_Q6K_PLANES && qtype != GGUF_Q6_K) return GGUF_ERR_UNSUPPORTED;
    if (K % block_values(qtype) != 0 || ld < K || ld % 8 != 0) return GGUF_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(out)) return GGUF_ERR_MISALIGNED;
    DeviceFacts* f = nullptr;
    int st = facts(&f);
    if (st != GGUF_OK) return st;
    return cuda_status(dequant_padded_launch(w, qtype, layout, N, K, out, odt, ld, f->num_sms, (cudaStream_t)stream));
}

int gguf_dense_gemm(const void* wdense, int wdt, int64_t ld, int64_t N, int64_t K, const void* x, int xdt, int64_t M,
                    const void* residual, void* y, int ydt, void* workspace, size_t ws_bytes, gguf_stream_t stream) {
    if (!wdense || !x || !y || N <= 0 || K <= 0 || M <= 0) return GGUF_ERR_INVALID_ARG;
    if ((wdt != GGUF_DT_F16 && wdt != GGUF_DT_BF16) || (xdt != GGUF_DT_F16 && xdt != GGUF_DT_BF16) ||
        !valid_dtype(ydt))
        return GGUF_ERR_UNSUPPORTED;
    if (K % 64 != 0 || ld < K || ld % 8 != 0) return GGUF_ERR_INVALID_ARG;
    if (!aligned16(wdense) || !aligned16(x) || !aligned16(y) || (residual && !aligned16(residual)))
        return GGUF_ERR_MISALIGNED;
    const size_t need = dense_workspace_bytes(N, K, M);
    if (need && (!workspace || ws_bytes < need)) return GGUF_ERR_WORKSPACE;
    if (workspace && !aligned16(workspace)) return GGUF_ERR_MISALIGNED;
    DeviceFacts* f = nullptr;
    int st = facts(&f);
    if (st != GGUF_OK) return st;
    return dense_gemm_run(wdense, wdt, ld, N, K, x, xdt, M, residual, y, ydt, workspace, f->num_sms, f->status,
                          (cudaStream_t)stream);
}

int gguf_mm_check_errors(gguf_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GGUF_ERR_CUDA;
    DeviceFacts* f = nullptr;
    int st = facts(&f);
    if (st != GGUF_OK) return st;
    int h = 0;
    if (cudaMemcpyFromSymbol(&h, g_status_word, sizeof(int)) != cudaSuccess) return GGUF_ERR_CUDA;
    if (h != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return GGUF_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return GGUF_ERR_CUDA;
    return h;
}

int gguf_mm_debug_moe_route(const int32_t* ids, int64_t entries, int64_t n_expert, int32_t* offsets,
                            int32_t* ntiles, int32_t* tiles, int64_t max_tiles, int32_t* rows, gguf_stream_t stream) {
    if (!ids || !offsets || !ntiles || !tiles || !rows || entries <= 0 || n_expert <= 0) return GGUF_ERR_INVALID_ARG;
    if (entries > INT32_MAX / 2 || n_expert > 4096) return GGUF_ERR_UNSUPPORTED;
    if (max_tiles < moe_max_tiles(n_expert, entries)) return GGUF_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(tiles) & 15u) || (reinterpret_cast<uintptr_t>(ids) & 3u)) return GGUF_ERR_MISALIGNED;
    DeviceFacts* f = nullptr;
    int st = facts(&f);
    if (st != GGUF_OK) return st;
    return moe_route_debug(ids, entries, n_expert, offsets, ntiles, reinterpret_cast<int4*>(tiles), max_tiles, rows,
                           (cudaStream_t)stream);
}

int gguf_mm_debug_timeout(int64_t spin_limit, gguf_stream_t stream) {
    if (spin_limit <= 0) return GGUF_ERR_INVALID_ARG;
    DeviceFacts* f = nullptr;
    int st = facts(&f);
    if (st != GGUF_OK) return st;
    timeout_probe_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((long long)spin_limit, f->status);
    return cuda_status(cudaGetLastError());
}

}  // extern "C"
