"""Decode GEMV (gguf_mm_gemv) against the int8-path oracle: integer intermediates
bit for bit for every GEMV kernel, outputs within the stated bounds, over
formats, layouts, shapes with ragged tails, activation/output dtypes and the
fused residual (OpenVINO PR #39119 "FullyConnectedGGUF", "Implementation",
GEMV row)."""
import numpy as np
import pytest
import torch

import gguf_quant_weight_gb300 as g
import gguf_synth as syn
from oracle import gguf_oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

QTYPES = [syn.Q8_0, syn.Q4_K, syn.Q5_K, syn.Q6_K]
QTYPES_32 = [syn.Q4_0, syn.Q4_1, syn.Q5_0, syn.Q5_1]
STAGED, DIRECT, TILE, PAIR, ROWLANE = 0, 1, 2, 3, 4


def _run_gemv(w_dev, qtype, layout, N, K, x, xdt, M, r, ydt, alias=False):
    y = U.guarded((M, N), U.TORCH_DT[ydt])
    nws = g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, qtype, N, K, M)
    ws = U.workspace(nws, 0xCD)
    rd = None if r is None else U.dev(r, ydt)
    if alias:
        y.t.copy_(rd)
        rd = y.t
    g.gguf_mm_gemv(w_dev, qtype, layout, N, K, U.dev(x, xdt), U.DT[xdt], M, rd, y.t, U.DT[ydt], ws.t, nws)
    torch.cuda.synchronize()
    y.check("y")
    ws.check("workspace")
    assert g.gguf_mm_check_errors() == 0
    return y.t


def _case(qtype, N, K, M, xdt="bf16", ydt="bf16", residual=True, layout=0, seed=0):
    rs = syn.rng(seed + 31 * qtype + 7 * N + K + M)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), xdt)
    r = syn.normal(rs, (M, N), ydt) if residual else None
    wd = U.dev(O.q6k_to_planes(w) if layout == g.GGUF_LAYOUT_Q6K_PLANES else w)
    y = _run_gemv(wd, qtype, layout, N, K, x, xdt, M, r, ydt)
    ref = O.gemv_int8_path(w, qtype, N, K, U.act_f32(x, xdt), None if r is None else U.act_f64(r, ydt))
    return U.host64(y), ref, w, x


def _terms(w, qtype, layout, N, K, x, xdt, M, kernel, residual=None):
    """Runs the debug build of the GEMV (forced kernel, f32 output); returns
    (kernel id that ran, qa, d_a, s, D, y) as numpy."""
    sub = 16 if qtype in (syn.Q6_K, syn.Q2_K, syn.Q3_K) else 32   # sub-block width of the dots
    qa = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    da = torch.zeros((M, K // 32), dtype=torch.float32, device="cuda")
    s = torch.zeros((M, K // 32), dtype=torch.int32, device="cuda")
    D = U.guarded((M, N, K // sub), torch.int32, fill=-999999)
    y = U.guarded((M, N), torch.float32)
    nws = g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, qtype, N, K, M)
    ws = U.workspace(nws, 0x5A)
    wd = U.dev(O.q6k_to_planes(w) if layout else w)
    ran = g.gguf_mm_debug_gemv_terms(wd, qtype, layout, N, K, U.dev(x, xdt), U.DT[xdt], M,
                                     None if residual is None else U.dev(residual, "f32"), y.t, g.GGUF_DT_F32,
                                     qa, da, s, D.t, ws.t, nws, kernel)
    torch.cuda.synchronize()
    for b, nm in ((D, "D"), (y, "y"), (ws, "workspace")):
        b.check(nm)
    assert g.gguf_mm_check_errors() == 0
    return ran, qa.cpu().numpy(), da.cpu().numpy(), s.cpu().numpy(), D.t.cpu().numpy(), U.host64(y.t)


def _assert_terms_exact(qtype, layout, N, K, M, kernel, seed=0, xdt="bf16", residual=False):
    rs = syn.rng(50 + qtype + 3 * M + N + K + seed)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), xdt)
    r = rs.standard_normal((M, N)).astype(np.float32) if residual else None
    ran, qa, da, s, D, y = _terms(w, qtype, layout, N, K, x, xdt, M, kernel, r)
    if kernel >= 0:
        assert ran == kernel, f"kernel {g.GEMV_KERNELS.get(ran)} ran, {g.GEMV_KERNELS[kernel]} was forced"
    y_ref, t = O.gemv_int8_path(w, qtype, N, K, U.act_f32(x, xdt), None if r is None else r.astype(np.float64),
                                return_terms=True)
    assert np.array_equal(qa, t["qa"])
    assert np.array_equal(da, t["d_a"])          # f32 bit patterns
    assert np.array_equal(s, t["s"])
    assert np.array_equal(D.astype(np.int64), t["D"]), f"D differs at {np.argwhere(D != t['D'])[:5]}"
    U.check_close(y, y_ref, "f32")
    return ran


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


# ---------------------------------------------------------------- integer terms, kernel by kernel

@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K])
@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(37, 1024), (300, 2048), (4096, 4096)])
def test_rowlane_kernel_integer_terms_bit_exact(qtype, M, N, K):
    # the decode workload's kernel (a lane per weight row), forced onto small
    # shapes too; ragged last CTA at N = 37 and 300
    _assert_terms_exact(qtype, 0, N, K, M, ROWLANE, residual=(M == 2))


@pytest.mark.parametrize("cluster", ["1", "2", "4"])
@pytest.mark.parametrize("M", [1, 2, 4])
@pytest.mark.parametrize("N,K", [(37, 1024), (129, 2048), (4096, 4096)])
def test_rowlane_cluster_sizes_integer_terms_bit_exact(cluster, M, N, K, monkeypatch):
    # CTAs in clusters of 1, 2 or 4 share the activation quantization (each
    # quantizes K / cluster of X into every image of the cluster); the grid is
    # rounded up to whole clusters at N = 37 and 129 (CTAs past N only quantize)
    monkeypatch.setenv("GGUF_MM_GEMV_CLUSTER", cluster)
    _assert_terms_exact(syn.Q5_K, 0, N, K, M, ROWLANE, seed=int(cluster), residual=(M != 2))


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K])
@pytest.mark.parametrize("N,K", [(37, 1024), (4096, 4096), (129, 768)])
def test_tile_kernel_integer_terms_bit_exact(qtype, N, K):
    _assert_terms_exact(qtype, 0, N, K, 1, TILE)


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K])
@pytest.mark.parametrize("M", [2, 3, 4])
def test_pair_kernel_integer_terms_bit_exact(qtype, M):
    _assert_terms_exact(qtype, 0, 41, 2048, M, PAIR)


@pytest.mark.parametrize("qtype,layout", [(syn.Q4_K, 0), (syn.Q5_K, 0), (syn.Q6_K, 1)])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_direct_kernel_integer_terms_bit_exact(qtype, layout, M):
    _assert_terms_exact(qtype, layout, 37, 768, M, DIRECT)


@pytest.mark.parametrize("qtype,layout", [(syn.Q8_0, 0), (syn.Q6_K, 0), (syn.Q6_K, 1), (syn.Q5_K, 0)])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_staged_kernel_integer_terms_bit_exact(qtype, layout, M):
    _assert_terms_exact(qtype, layout, 37, 768, M, STAGED)


@pytest.mark.parametrize("qtype", QTYPES_32)
@pytest.mark.parametrize("N,K,M", [(37, 768, 1), (37, 96, 3), (300, 2048, 8), (129, 4352, 2)])
def test_32_value_formats_integer_terms_bit_exact(qtype, N, K, M):
    # Q4_0 / Q4_1 / Q5_0 / Q5_1 on the staged kernel: dots of (q - 8), (q5 - 16)
    # or the unsigned codes, bit for bit; K need only be a multiple of 32
    assert _assert_terms_exact(qtype, 0, N, K, M, -1, residual=(M == 2)) == STAGED


@pytest.mark.parametrize("qtype", [syn.Q2_K, syn.Q3_K])
@pytest.mark.parametrize("N,K,M", [(37, 768, 1), (37, 256, 3), (300, 2048, 8), (129, 4352, 2)])
def test_2_and_3_bit_kquants_integer_terms_bit_exact(qtype, N, K, M):
    # Q2_K / Q3_K on the staged kernel: 16-value sub-block dots of q2 and of q3
    # (the unsigned q3 + 4 dot less 4 times the sub-block's code sum), bit for bit
    assert _assert_terms_exact(qtype, 0, N, K, M, -1, residual=(M == 2)) == STAGED


@pytest.mark.parametrize("qtype", [syn.Q2_K, syn.Q3_K])
@pytest.mark.parametrize("N,K", [(1, 256), (3, 512), (128, 1024), (200, 4352)])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_2_and_3_bit_kquants_outputs(qtype, N, K, M):
    got, ref, _, _ = _case(qtype, N, K, M)
    U.check_close(got, ref, "bf16", what=f"q{qtype} N{N} K{K} M{M}")


@pytest.mark.parametrize("qtype", QTYPES_32)
@pytest.mark.parametrize("N,K", [(1, 32), (3, 512), (128, 1024), (129, 800)])
@pytest.mark.parametrize("M", [1, 4])
def test_32_value_formats_outputs(qtype, N, K, M):
    got, ref, _, _ = _case(qtype, N, K, M)
    U.check_close(got, ref, "bf16", what=f"q{qtype} N{N} K{K} M{M}")


@pytest.mark.parametrize("M", [1, 2, 4])
def test_decode_workload_plan_is_rowlane_and_bit_exact(M):
    # the plan's own choice for Q5_K 4096 x 4096 (no forcing): the row-lane kernel
    assert g.gguf_mm_gemv_kernel(syn.Q5_K, 0, 4096, 4096, M) == ROWLANE
    assert _assert_terms_exact(syn.Q5_K, 0, 4096, 4096, M, -1, seed=1001) == ROWLANE


def test_small_workload_plan_and_terms():
    # Q6_K 256 x 1024, f32 activations: the staged kernel
    assert _assert_terms_exact(syn.Q6_K, 0, 256, 1024, 1, -1, xdt="f32") == g.gguf_mm_gemv_kernel(
        syn.Q6_K, 0, 256, 1024, 1, g.GGUF_DT_F32)


# ---------------------------------------------------------------- outputs

@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("N,K", [(1, 256), (3, 512), (128, 1024), (129, 768), (200, 4352)])
@pytest.mark.parametrize("M", [1, 3, 8])
def test_gemv_small_shapes(qtype, N, K, M):
    got, ref, _, _ = _case(qtype, N, K, M)
    U.check_close(got, ref, "bf16", what=f"q{qtype} N{N} K{K} M{M}")


@pytest.mark.parametrize("M", [1, 2, 4, 5, 6, 7])
@pytest.mark.parametrize("qtype", [syn.Q5_K, syn.Q6_K])
def test_gemv_all_row_counts(qtype, M):
    got, ref, _, _ = _case(qtype, 130, 1024, M)
    U.check_close(got, ref, "bf16")


@pytest.mark.parametrize("xdt,ydt", [("f32", "f32"), ("f16", "f16"), ("bf16", "f32"), ("f32", "bf16")])
@pytest.mark.parametrize("qtype", QTYPES)
def test_gemv_dtypes(qtype, xdt, ydt):
    got, ref, _, _ = _case(qtype, 96, 512, 2, xdt=xdt, ydt=ydt)
    U.check_close(got, ref, ydt)


@pytest.mark.parametrize("N,K", [(64, 512), (33, 1280), (256, 1024)])
def test_gemv_q6k_planes_equals_blocks(N, K):
    got_p, ref, _, _ = _case(syn.Q6_K, N, K, 2, layout=g.GGUF_LAYOUT_Q6K_PLANES)
    got_b, _, _, _ = _case(syn.Q6_K, N, K, 2, layout=0)
    U.check_close(got_p, ref, "bf16")
    assert np.array_equal(got_p, got_b)          # same arithmetic, same order


@pytest.mark.parametrize("N,M", [(160, 3), (4096, 1), (4096, 4)])
def test_gemv_residual_may_alias_output(N, M):
    rs = syn.rng(3 + M)
    K = 1024 if N < 4096 else 4096
    w = syn.weight_blocks(rs, syn.Q5_K, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    r = syn.normal(rs, (M, N), "bf16")
    y = _run_gemv(U.dev(w), syn.Q5_K, 0, N, K, x, "bf16", M, r, "bf16", alias=True)
    ref = O.gemv_int8_path(w, syn.Q5_K, N, K, U.act_f32(x, "bf16"), U.act_f64(r, "bf16"))
    U.check_close(U.host64(y), ref, "bf16")


@pytest.mark.parametrize("qtype,N,K,M,ydt,residual", [
    (syn.Q5_K, 4096, 4096, 1, "bf16", True), (syn.Q5_K, 4096, 4096, 4, "bf16", True),
    (syn.Q5_K, 300, 1024, 2, "f32", False), (syn.Q8_0, 200, 768, 3, "bf16", True), (syn.Q4_0, 37, 512, 8, "f32", True)])
def test_gemv_from_host_buffers(qtype, N, K, M, ydt, residual):
    # gguf_mm_gemv_host: copy in, the GEMV, copy out, in one call on pinned host
    # buffers; y_host equals the device-buffer call's output bit for bit
    rs = syn.rng(17 + qtype + M + N)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    r = syn.normal(rs, (M, N), ydt) if residual else None
    wd = U.dev(w)
    tdt = U.TORCH_DT[ydt]
    xh = torch.from_numpy(x.copy()).view(torch.bfloat16).pin_memory()
    rh = None if r is None else torch.from_numpy(r.copy()).view(tdt).pin_memory()
    yh = torch.full((M, N), float("nan"), dtype=tdt).pin_memory()
    xd = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    rd = None if r is None else torch.empty((M, N), dtype=tdt, device="cuda")
    yd = U.guarded((M, N), tdt)
    nws = g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, qtype, N, K, M)
    ws = U.workspace(nws, 0xCD)
    g.gguf_mm_gemv_host(wd, qtype, 0, N, K, xh, xd, g.GGUF_DT_BF16, M, rh, rd, yh, yd.t, U.DT[ydt], ws.t, nws)
    torch.cuda.synchronize()
    yd.check("y")
    ws.check("workspace")
    assert g.gguf_mm_check_errors() == 0
    y_dev_call = _run_gemv(wd, qtype, 0, N, K, x, "bf16", M, r, ydt)
    assert torch.equal(yh.view(torch.int16 if ydt == "bf16" else torch.int32),
                       y_dev_call.cpu().view(torch.int16 if ydt == "bf16" else torch.int32))
    ref = O.gemv_int8_path(w, qtype, N, K, U.act_f32(x, "bf16"), None if r is None else U.act_f64(r, ydt))
    U.check_close(yh.double().numpy(), ref, ydt)


def test_gemv_config_q6k_256x1024_f32():
    # the small decode workload: Q6_K N=256 K=1024 M=1, f32 in / f32 out
    cfg = syn.CONFIGS["q6k_gemv_256x1024"]
    rs = syn.rng(cfg["seed"])
    w = syn.weight_blocks(rs, syn.Q6_K, 256, 1024)
    x = syn.normal(rs, (1, 1024), "f32")
    y = _run_gemv(U.dev(w), syn.Q6_K, 0, 256, 1024, x, "f32", 1, None, "f32")
    ref = O.gemv_int8_path(w, syn.Q6_K, 256, 1024, x)
    U.check_close(U.host64(y), ref, "f32")


@pytest.mark.parametrize("ydt", ["bf16", "f32"])
@pytest.mark.parametrize("M", [1, 2, 4])
def test_gemv_config_q5k_4096x4096_residual(M, ydt):
    cfg = syn.CONFIGS["q5k_gemv_4096x4096_res"]
    rs = syn.rng(cfg["seed"] + M)
    N = K = 4096
    w = syn.weight_blocks(rs, syn.Q5_K, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    r = syn.normal(rs, (M, N), ydt)
    y = _run_gemv(U.dev(w), syn.Q5_K, 0, N, K, x, "bf16", M, r, ydt)
    ref = O.gemv_int8_path(w, syn.Q5_K, N, K, U.act_f32(x, "bf16"), U.act_f64(r, ydt))
    U.check_close(U.host64(y), ref, ydt)
    # the gap to the exact (unquantized-activation) matmul is reported, not gated
    exact = O.matmul_exact(U.act_f64(x, "bf16"), O.dequant(w, syn.Q5_K, N, K), U.act_f64(r, ydt))
    gap = np.max(np.abs(U.host64(y) - exact)) / np.max(np.abs(exact))
    print(f"Q5_K 4096x4096 M={M} {ydt}: gap to exact matmul {gap:.2e} of max|ref|")


def test_gemv_status_ok_after_runs():
    assert g.gguf_mm_check_errors() == 0


# ---------------------------------------------------------------- the activation quantizer's edge cases

def _quantizer_terms(qtype, N, K, x, kernel=-1):
    M = x.shape[0]
    w = syn.weight_blocks(syn.rng(9), qtype, N, K)
    with np.errstate(all="ignore"):
        ran, qa, da, s, _, _ = _terms(w, qtype, 0, N, K, x, "f32", M, kernel)
        rqa, rda, rs_ = O.quantize_act_q8(x)
    assert np.array_equal(qa, rqa)
    assert np.array_equal(da, rda, equal_nan=True)
    assert np.array_equal(s, rs_)
    return ran, qa, da


@pytest.mark.parametrize("qtype,kernel", [(syn.Q4_K, ROWLANE), (syn.Q4_K, TILE), (syn.Q6_K, -1)])
def test_gemv_activation_quantizer_edge_blocks(qtype, kernel):
    # zero block, constant block, exact grid multiples and .5 ties; each of the
    # kernels that quantize inside the GEMV, and the stand-alone quantizer
    K = 256
    rs = syn.rng(9)
    x = np.zeros((2, K), np.float32)
    x[0, 32:64] = 0.3
    x[0, 64:96] = np.arange(32) - 16.0
    x[0, 64] = 127.0
    x[0, 96:128] = 2.5
    x[0, 96] = 127.0
    x[1] = rs.standard_normal(K).astype(np.float32) * 1e-30
    ran, qa, da = _quantizer_terms(qtype, 40, K, x[:1] if kernel == TILE else x, kernel)
    assert np.all(qa[0, :32] == 0) and da[0, 0] == 0


@pytest.mark.parametrize("qtype,kernel", [(syn.Q4_K, ROWLANE), (syn.Q4_K, TILE), (syn.Q6_K, -1)])
def test_gemv_activation_quantizer_non_finite_and_extreme_blocks(qtype, kernel):
    # the same rule as the oracle on every input: ties away from zero over a
    # whole range of halves, a NaN block (NaN scale, every code -127), an inf
    # block (scale inf, codes 0 except -127 at the inf), a block whose 1/d_a
    # overflows (every code 127), one just above that limit, and huge values
    K = 512
    rs = syn.rng(11)
    x = np.zeros((2, K), np.float32)
    x[0, 0] = 127.0
    x[0, 1:32] = np.arange(-15, 16) + 0.5
    x[0, 32:64] = np.linspace(-3, 3, 32)
    x[0, 37] = np.nan
    x[0, 64:96] = 1.0
    x[0, 72] = np.inf
    x[0, 96:128] = 1e-39
    x[0, 128:160] = 4e-37 * rs.standard_normal(32)
    x[0, 160:192] = 3.0e38 * np.sign(rs.standard_normal(32))
    x[0, 192:224] = -np.inf
    x[1] = rs.standard_normal(K).astype(np.float32)
    x[1, 256:288] = np.float32(127.0) * (np.arange(32) % 2) - 0.5 * (np.arange(32) % 3)
    _quantizer_terms(qtype, 40, K, x[:1] if kernel == TILE else x, kernel)


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K])
@pytest.mark.parametrize("N,K", [(300, 2048), (1000, 4096), (77, 8192)])
@pytest.mark.parametrize("M", [2, 3, 4])
def test_gemv_m2_to_m4_shapes(qtype, N, K, M):
    got, ref, _, _ = _case(qtype, N, K, M)
    U.check_close(got, ref, "bf16", what=f"q{qtype} N{N} K{K} M{M}")
