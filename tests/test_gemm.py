"""Fused prefill GEMM (gguf_mm_gemm, path FUSED): weights decoded in the kernel
to f16 and multiplied on tcgen05 tensor cores, against the exact f64 oracle
(OpenVINO PR #39119, "Implementation", DPAS prefill row)."""
import functools

import numpy as np
import pytest
import torch

import gguf_quant_weight_gb300 as g
import gguf_synth as syn
from oracle import gguf_oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


def _launch(wd, qtype, layout, N, K, x, xdt, M, r, ydt, path=g.GGUF_PATH_FUSED, ws_fill=0x3C):
    y = U.guarded((M, N), U.TORCH_DT[ydt])
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qtype, N, K, M)
    ws = U.workspace(ws_bytes, ws_fill)
    g.gguf_mm_gemm(wd, qtype, layout, N, K, U.dev(x, xdt), U.DT[xdt], M, None if r is None else U.dev(r, ydt),
                   y.t, U.DT[ydt], ws.t, ws_bytes, path)
    torch.cuda.synchronize()
    y.check("y")
    ws.check("workspace")
    assert g.gguf_mm_check_errors() == 0
    return U.host64(y.t)


def _gemm(qtype, N, K, M, layout=0, ydt="bf16", xdt="bf16", residual=True, seed=0, path=g.GGUF_PATH_FUSED,
          rows=None):
    rs = syn.rng(seed + 7 * N + K + 3 * M + qtype)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), xdt)
    r = syn.normal(rs, (M, N), ydt) if residual else None
    wd = U.dev(O.q6k_to_planes(w) if layout else w)
    got = _launch(wd, qtype, layout, N, K, x, xdt, M, r, ydt, path)
    sel = slice(None) if rows is None else rows
    ref = O.matmul_exact(U.act_f64(x[sel], xdt), O.dequant(w, qtype, N, K),
                         None if r is None else U.act_f64(r[sel], ydt))
    return got[sel], ref


@pytest.mark.parametrize("qtype,K", [(syn.Q8_0, 256), (syn.Q8_0, 1024), (syn.Q4_K, 256), (syn.Q4_K, 768),
                                     (syn.Q5_K, 512), (syn.Q5_K, 1280), (syn.Q6_K, 2048)])
@pytest.mark.parametrize("N,M", [(128, 16), (200, 40), (384, 130), (130, 300)])
def test_fused_small(qtype, K, N, M):
    got, ref = _gemm(qtype, N, K, M)
    U.check_close(got, ref, "bf16", what=f"q{qtype} N{N} K{K} M{M}")


@pytest.mark.parametrize("qtype", [syn.Q4_0, syn.Q4_1, syn.Q5_0, syn.Q5_1])
@pytest.mark.parametrize("N,K,M", [(128, 256, 16), (200, 768, 40), (384, 1024, 130), (130, 2048, 300)])
def test_fused_32_value_formats(qtype, N, K, M):
    got, ref = _gemm(qtype, N, K, M)
    U.check_close(got, ref, "bf16", what=f"q{qtype} N{N} K{K} M{M}")


@pytest.mark.parametrize("qtype,K", [(syn.Q2_K, 1024), (syn.Q2_K, 4096), (syn.Q3_K, 2048), (syn.Q3_K, 4096)])
@pytest.mark.parametrize("N,M", [(128, 16), (200, 40), (384, 130), (130, 300)])
def test_fused_2_and_3_bit_kquants(qtype, K, N, M):
    # raw rows staged by TMA from their 16-byte boundary (84- and 110-byte blocks)
    got, ref = _gemm(qtype, N, K, M)
    U.check_close(got, ref, "bf16", what=f"q{qtype} N{N} K{K} M{M}")


@pytest.mark.parametrize("qtype", [syn.Q2_K, syn.Q3_K])
def test_fused_2_and_3_bit_kquants_f32_out_split_k(qtype):
    got, ref = _gemm(qtype, 256, 4096, 48, ydt="f32")
    U.check_close(got, ref, "f32", rel=2e-3)


@pytest.mark.parametrize("qtype", [syn.Q4_0, syn.Q4_1, syn.Q5_0, syn.Q5_1])
def test_fused_32_value_formats_f32_out_split_k(qtype):
    # few row tiles: the plan splits K; f32 output holds the bound raw
    got, ref = _gemm(qtype, 256, 4096, 48, ydt="f32")
    U.check_close(got, ref, "f32", rel=2e-3)


@pytest.mark.parametrize("N,M", [(128, 8), (256, 64), (200, 257)])
def test_fused_q6k_planes(N, M):
    got, ref = _gemm(syn.Q6_K, N, 2048, M, layout=1)
    U.check_close(got, ref, "bf16")


@pytest.mark.parametrize("ydt", ["f32", "f16"])
@pytest.mark.parametrize("qtype", [syn.Q5_K, syn.Q8_0, syn.Q4_K, syn.Q6_K])
def test_fused_out_dtypes(qtype, ydt):
    got, ref = _gemm(qtype, 256, 512 if qtype != syn.Q6_K else 2048, 48, ydt=ydt)
    U.check_close(got, ref, ydt, rel=2e-3)


def test_fused_f16_activations_no_residual():
    got, ref = _gemm(syn.Q4_K, 256, 512, 33, xdt="f16", residual=False)
    U.check_close(got, ref, "bf16")


@pytest.mark.parametrize("M", [9, 40, 300])
def test_fused_f32_activations(M):
    # f32 activations are converted to f16 row by row (one rounding each)
    got, ref = _gemm(syn.Q5_K, 256, 1024, M, xdt="f32", ydt="f32")
    U.check_close(got, ref, "f32", rel=2e-3)


@pytest.mark.parametrize("qtype,layout,N,K", [(syn.Q5_K, 0, 256, 1024), (syn.Q8_0, 0, 9000, 1024),
                                              (syn.Q6_K, 0, 512, 2048)])
@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_auto_path_follows_the_crossover(qtype, layout, N, K, xdt):
    # AUTO's choice for every row count around the crossover, and the output
    # of the path it chose: the int8-path oracle for the GEMV, the exact one
    # for the fused GEMM
    rs = syn.rng(3 + qtype)
    w = syn.weight_blocks(rs, qtype, N, K)
    seen = set()
    for M in range(1, 11):
        path = g.gguf_mm_auto_path(qtype, layout, N, K, M, U.DT[xdt])
        assert path in (g.GGUF_PATH_GEMV, g.GGUF_PATH_FUSED)
        if M > 8:
            assert path == g.GGUF_PATH_FUSED
        seen.add(path)
        x = syn.normal(rs, (M, K), xdt)
        got = _launch(U.dev(w), qtype, layout, N, K, x, xdt, M, None, "f32", path=g.GGUF_PATH_AUTO)
        if path == g.GGUF_PATH_GEMV:
            U.check_close(got, O.gemv_int8_path(w, qtype, N, K, U.act_f32(x, xdt)), "f32")
        else:
            U.check_close(got, O.matmul_exact(U.act_f64(x, xdt), O.dequant(w, qtype, N, K)), "f32", rel=2e-3)
    assert seen == {g.GGUF_PATH_GEMV, g.GGUF_PATH_FUSED}


# ---------------------------------------------------------------- the prefill workloads at full size

@functools.lru_cache(maxsize=1)
def _weights(qtype, N, K, seed):
    w = syn.weight_blocks(syn.rng(seed + qtype), qtype, N, K)
    return w, O.dequant(w, qtype, N, K)


def _full(qtype, layout, N, K, M, seed, ydt="bf16"):
    w, w64 = _weights(qtype, N, K, seed)
    rs = syn.rng(seed + M)
    x = syn.normal(rs, (M, K), "bf16")
    wd = U.dev(O.q6k_to_planes(w) if layout else w)
    got = _launch(wd, qtype, layout, N, K, x, "bf16", M, None, ydt)
    rows = np.unique(np.concatenate([np.arange(0, M, max(1, M // 5)), [M - 1]]))
    ref = O.matmul_exact(U.act_f64(x[rows], "bf16"), w64)
    return got[rows], ref


@pytest.mark.parametrize("M", [8, 64, 128, 256, 512, 2048])
@pytest.mark.parametrize("qtype,layout", [(syn.Q6_K, 0), (syn.Q6_K, 1), (syn.Q5_K, 0), (syn.Q4_K, 0),
                                          (syn.Q8_0, 0)])
def test_fused_config_14336x4096(qtype, layout, M):
    # the prefill workload (every row count); sampled activation rows, all 14336 outputs
    got, ref = _full(qtype, layout, 14336, 4096, M, 1002)
    U.check_close(got, ref, "bf16", what=f"q{qtype}/{layout} M{M}")


@pytest.mark.parametrize("M", [512, 2048])
@pytest.mark.parametrize("qtype,layout", [(syn.Q5_K, 0), (syn.Q6_K, 1)])
def test_fused_config_14336x4096_f32_out(qtype, layout, M):
    # the same with f32 output: the bound holds with nothing granted for rounding
    got, ref = _full(qtype, layout, 14336, 4096, M, 1002, ydt="f32")
    U.check_close(got, ref, "f32", rel=2e-3)


@pytest.mark.parametrize("M", [128, 512, 4096])
def test_fused_config_q8_0_2048x8192(M):
    got, ref = _full(syn.Q8_0, 0, 2048, 8192, M, 1003)
    U.check_close(got, ref, "bf16")


def test_fused_rejects_q6k_rows_without_16_byte_stride():
    w = torch.zeros(256 * 210, dtype=torch.uint8, device="cuda")
    x = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.GGUFError) as e:
        g.gguf_mm_gemm(w, syn.Q6_K, 0, 256, 256, x, g.GGUF_DT_BF16, 16, None, y, g.GGUF_DT_BF16, ws, 1 << 16,
                       g.GGUF_PATH_FUSED)
    assert e.value.status == g.GGUF_ERR_UNSUPPORTED


@pytest.mark.parametrize("qtype,N,K,M", [(syn.Q4_K, 256, 4096, 40), (syn.Q4_K, 14336, 1024, 512)])
def test_fused_split_k_residual_exact_and_deterministic(qtype, N, K, M):
    # 2 row tiles at K = 4096 leave most SMs idle, so the plan splits every
    # tile's K; 224 tiles on 152 SMs keep one round whole and split the other
    # 72 into K halves.  Stale workspace bytes (tickets included) must not
    # matter, two runs agree bit for bit, and both match the oracle.
    rs = syn.rng(4242 + N)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    r = syn.normal(rs, (M, N), "bf16")
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qtype, N, K, M)
    if N == 256:
        assert ws_bytes > M * K * 2 + M * 4   # room for the partial tiles
    outs = [_launch(U.dev(w), qtype, 0, N, K, x, "bf16", M, r, "bf16", ws_fill=fill) for fill in (0x00, 0xFF)]
    assert np.array_equal(outs[0], outs[1])
    ref = O.matmul_exact(U.act_f64(x, "bf16"), O.dequant(w, qtype, N, K), U.act_f64(r, "bf16"))
    U.check_close(outs[0], ref, "bf16")


def _range_rows(rs, M, K):
    """Activation rows of every magnitude: f16's range is 6.1e-5 .. 65504."""
    x32 = rs.standard_normal((M, K)).astype(np.float32)
    x32[0] *= 3e5
    x32[1] *= 1e20
    x32[2] *= 1e-7
    x32[3, ::7] *= 1e5          # a few large values in an ordinary row
    x32[4] *= 1e-30
    return x32


@pytest.mark.parametrize("xdt", ["bf16", "f32"])
@pytest.mark.parametrize("qtype,N,K,M", [(syn.Q4_K, 256, 1024, 24), (syn.Q6_K, 14336, 2048, 512),
                                         (syn.Q8_0, 2048, 8192, 128)])
def test_fused_activation_rows_beyond_f16_range(qtype, N, K, M, xdt):
    # each activation row is converted to f16 scaled by a power of two that
    # puts its largest magnitude in [2^14, 2^15); the epilogue scales its sums
    # back.  Checked row by row, each against its own scale (f32 output).
    rs = syn.rng(61 + qtype + M)
    w = syn.weight_blocks(rs, qtype, N, K)
    x32 = _range_rows(rs, M, K)
    x = syn.f32_to_bf16_bits(x32) if xdt == "bf16" else x32
    got = _launch(U.dev(w), qtype, 0, N, K, x, xdt, M, None, "f32")
    rows = np.array([0, 1, 2, 3, 4, 5, M - 1])
    ref = O.matmul_exact(U.act_f64(x[rows], xdt), O.dequant(w, qtype, N, K))
    for i, m in enumerate(rows):
        U.check_close(got[m], ref[i], "f32", rel=2e-3, what=f"row {m}")
