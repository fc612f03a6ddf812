"""Decode GEMV (gguf_mm_gemv) against the int8-path oracle: integer intermediates
bit for bit, outputs within the stated bounds, over formats, layouts, shapes
with ragged tails, activation/output dtypes and the fused residual."""
import numpy as np
import pytest
import torch

import gguf_quant_weight_gb300 as g
import gguf_synth as syn
from oracle import gguf_oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

QTYPES = [syn.Q8_0, syn.Q4_K, syn.Q5_K, syn.Q6_K]


def _run_gemv(w_dev, qtype, layout, N, K, x, xdt, M, r, ydt):
    y = torch.empty((M, N), dtype=U.TORCH_DT[ydt], device="cuda")
    ws, ws_bytes = U.gemv_workspace(M, K)
    g.gguf_mm_gemv(w_dev, qtype, layout, N, K, U.dev(x, xdt), U.DT[xdt], M,
                   None if r is None else U.dev(r, ydt), y, U.DT[ydt], ws, ws_bytes)
    torch.cuda.synchronize()
    return y


def _case(qtype, N, K, M, xdt="bf16", ydt="bf16", residual=True, layout=0, seed=0):
    rs = syn.rng(seed + 31 * qtype + 7 * N + K + M)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), xdt)
    r = syn.normal(rs, (M, N), ydt) if residual else None
    wd = U.dev(w)
    if layout == g.GGUF_LAYOUT_Q6K_PLANES:
        wd = U.dev(O.q6k_to_planes(w))
    y = _run_gemv(wd, qtype, layout, N, K, x, xdt, M, r, ydt)
    ref = O.gemv_int8_path(w, qtype, N, K, U.act_f32(x, xdt), None if r is None else U.act_f64(r, ydt))
    return U.host64(y), ref, w, x


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


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


def test_gemv_residual_may_alias_output():
    rs = syn.rng(3)
    N, K, M = 160, 1024, 3
    w = syn.weight_blocks(rs, syn.Q5_K, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    r = syn.normal(rs, (M, N), "bf16")
    y = U.dev(r, "bf16").clone()
    ws, ws_bytes = U.gemv_workspace(M, K)
    g.gguf_mm_gemv(U.dev(w), syn.Q5_K, 0, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, y, y, g.GGUF_DT_BF16,
                   ws, ws_bytes)
    torch.cuda.synchronize()
    ref = O.gemv_int8_path(w, syn.Q5_K, N, K, U.act_f32(x, "bf16"), U.act_f64(r, "bf16"))
    U.check_close(U.host64(y), ref, "bf16")


@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("layout", [0, 1])
def test_gemv_integer_terms_bit_exact(qtype, layout):
    if layout == 1 and qtype != syn.Q6_K:
        pytest.skip("planes exist for Q6_K only")
    rs = syn.rng(50 + qtype)
    N, K, M = 37, 768, 3
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    sub = 16 if qtype == syn.Q6_K else 32
    qa = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    da = torch.zeros((M, K // 32), dtype=torch.float32, device="cuda")
    s = torch.zeros((M, K // 32), dtype=torch.int32, device="cuda")
    D = torch.full((M, N, K // sub), -999999, dtype=torch.int32, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    wd = U.dev(O.q6k_to_planes(w) if layout else w)
    g.gguf_mm_debug_gemv_terms(wd, qtype, layout, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, y, g.GGUF_DT_F32,
                               qa, da, s, D)
    torch.cuda.synchronize()
    y_ref, terms = O.gemv_int8_path(w, qtype, N, K, U.act_f32(x, "bf16"), return_terms=True)
    assert np.array_equal(qa.cpu().numpy(), terms["qa"])
    assert np.array_equal(da.cpu().numpy(), terms["d_a"])          # f32 bit patterns
    assert np.array_equal(s.cpu().numpy(), terms["s"])
    assert np.array_equal(D.cpu().numpy().astype(np.int64), terms["D"])
    U.check_close(U.host64(y), y_ref, "f32")


def test_gemv_activation_quantizer_edge_blocks():
    # zero block, constant block, exact grid multiples and .5 ties
    N, K, M = 8, 256, 2
    rs = syn.rng(9)
    w = syn.weight_blocks(rs, syn.Q4_K, N, K)
    x = np.zeros((M, K), np.float32)
    x[0, 32:64] = 0.3
    x[0, 64:96] = np.arange(32) - 16.0
    x[0, 64] = 127.0
    x[0, 96:128] = 2.5
    x[0, 96] = 127.0
    x[1] = rs.standard_normal(K).astype(np.float32) * 1e-30
    qa = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    da = torch.zeros((M, K // 32), dtype=torch.float32, device="cuda")
    s = torch.zeros((M, K // 32), dtype=torch.int32, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g.gguf_mm_debug_gemv_terms(U.dev(w), syn.Q4_K, 0, N, K, U.dev(x), g.GGUF_DT_F32, M, y, g.GGUF_DT_F32,
                               qa, da, s, None)
    torch.cuda.synchronize()
    rqa, rda, rs_ = O.quantize_act_q8(x)
    assert np.array_equal(qa.cpu().numpy(), rqa)
    assert np.array_equal(da.cpu().numpy(), rda)
    assert np.array_equal(s.cpu().numpy(), rs_)
    assert np.all(qa.cpu().numpy()[0, :32] == 0) and da.cpu().numpy()[0, 0] == 0


def test_gemv_config_q6k_256x1024_f32():
    # the small decode workload: Q6_K N=256 K=1024 M=1, f32 in / f32 out
    cfg = syn.CONFIGS["q6k_gemv_256x1024"]
    rs = syn.rng(cfg["seed"])
    w = syn.weight_blocks(rs, syn.Q6_K, 256, 1024)
    x = syn.normal(rs, (1, 1024), "f32")
    y = _run_gemv(U.dev(w), syn.Q6_K, 0, 256, 1024, x, "f32", 1, None, "f32")
    ref = O.gemv_int8_path(w, syn.Q6_K, 256, 1024, x)
    U.check_close(U.host64(y), ref, "f32")


@pytest.mark.parametrize("M", [1, 2, 4])
def test_gemv_config_q5k_4096x4096_residual(M):
    cfg = syn.CONFIGS["q5k_gemv_4096x4096_res"]
    rs = syn.rng(cfg["seed"] + M)
    N = K = 4096
    w = syn.weight_blocks(rs, syn.Q5_K, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    r = syn.normal(rs, (M, N), "bf16")
    y = _run_gemv(U.dev(w), syn.Q5_K, 0, N, K, x, "bf16", M, r, "bf16")
    ref = O.gemv_int8_path(w, syn.Q5_K, N, K, U.act_f32(x, "bf16"), U.act_f64(r, "bf16"))
    U.check_close(U.host64(y), ref, "bf16")
    # the gap to the exact (unquantized-activation) matmul is reported, not gated
    exact = O.matmul_exact(U.act_f64(x, "bf16"), O.dequant(w, syn.Q5_K, N, K), U.act_f64(r, "bf16"))
    gap = np.max(np.abs(U.host64(y) - exact)) / np.max(np.abs(exact))
    print(f"Q5_K 4096x4096 M={M}: gap to exact matmul {gap:.2e} of max|ref|")


def test_gemv_status_ok_after_runs():
    assert g.gguf_mm_check_errors() == 0


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q6_K])
def test_gemv_activation_quantizer_non_finite_and_extreme_blocks(qtype):
    # the same rule as the oracle on every input: ties away from zero over a
    # whole range of halves, a NaN block (NaN scale, every code -127), an inf
    # block (scale inf, codes 0 except -127 at the inf), a block whose 1/d_a
    # overflows (every code 127), one just above that limit, and huge values.
    # Q4_K runs the quantizer inside the GEMV kernel, raw Q6_K the stand-alone one.
    N, K, M = 8, 512, 2
    rs = syn.rng(11)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = np.zeros((M, K), np.float32)
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
    qa = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    da = torch.zeros((M, K // 32), dtype=torch.float32, device="cuda")
    s = torch.zeros((M, K // 32), dtype=torch.int32, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g.gguf_mm_debug_gemv_terms(U.dev(w), qtype, 0, N, K, U.dev(x), g.GGUF_DT_F32, M, y, g.GGUF_DT_F32,
                               qa, da, s, None)
    torch.cuda.synchronize()
    with np.errstate(all="ignore"):
        rqa, rda, rs_ = O.quantize_act_q8(x)
    assert np.array_equal(qa.cpu().numpy(), rqa)
    assert np.array_equal(da.cpu().numpy(), rda, equal_nan=True)
    assert np.array_equal(s.cpu().numpy(), rs_)


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K])
@pytest.mark.parametrize("N,K", [(300, 2048), (1000, 4096), (77, 8192)])
@pytest.mark.parametrize("M", [2, 3, 4])
def test_gemv_pair_kernel_shapes(qtype, N, K, M):
    # K a multiple of 2048 and 2..4 rows: the kernel that keeps each lane's
    # 64-value slice of the activation codes in registers
    got, ref, _, _ = _case(qtype, N, K, M)
    U.check_close(got, ref, "bf16", what=f"q{qtype} N{N} K{K} M{M}")


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K])
def test_gemv_pair_kernel_integer_terms_bit_exact(qtype):
    rs = syn.rng(70 + qtype)
    N, K, M = 41, 2048, 3
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    qa = torch.zeros((M, K), dtype=torch.int8, device="cuda")
    da = torch.zeros((M, K // 32), dtype=torch.float32, device="cuda")
    s = torch.zeros((M, K // 32), dtype=torch.int32, device="cuda")
    D = torch.full((M, N, K // 32), -999999, dtype=torch.int32, device="cuda")
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g.gguf_mm_debug_gemv_terms(U.dev(w), qtype, 0, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, y, g.GGUF_DT_F32,
                               qa, da, s, D)
    torch.cuda.synchronize()
    y_ref, terms = O.gemv_int8_path(w, qtype, N, K, U.act_f32(x, "bf16"), return_terms=True)
    assert np.array_equal(qa.cpu().numpy(), terms["qa"])
    assert np.array_equal(da.cpu().numpy(), terms["d_a"])
    assert np.array_equal(s.cpu().numpy(), terms["s"])
    assert np.array_equal(D.cpu().numpy().astype(np.int64), terms["D"])
    U.check_close(U.host64(y), y_ref, "f32")
