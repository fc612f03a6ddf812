"""Fused prefill GEMM (gguf_mm_gemm, path FUSED): weights decoded in the kernel
to f16 and multiplied on tcgen05 tensor cores, against the exact f64 oracle
(OpenVINO PR #39119, "Implementation", DPAS prefill row)."""
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


def _gemm(qtype, N, K, M, layout=0, ydt="bf16", xdt="bf16", residual=True, seed=0, path=g.GGUF_PATH_FUSED,
          rows=None):
    rs = syn.rng(seed + 7 * N + K + 3 * M + qtype)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), xdt)
    r = syn.normal(rs, (M, N), ydt) if residual else None
    wd = U.dev(O.q6k_to_planes(w) if layout else w)
    y = torch.empty((M, N), dtype=U.TORCH_DT[ydt], device="cuda")
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qtype, N, K, M)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    g.gguf_mm_gemm(wd, qtype, layout, N, K, U.dev(x, xdt), U.DT[xdt], M, None if r is None else U.dev(r, ydt), y,
                   U.DT[ydt], ws, ws_bytes, path)
    torch.cuda.synchronize()
    assert g.gguf_mm_check_errors() == 0
    sel = slice(None) if rows is None else rows
    ref = O.matmul_exact(U.act_f64(x[sel], xdt), O.dequant(w, qtype, N, K),
                         None if r is None else U.act_f64(r[sel], ydt))
    return U.host64(y)[sel], ref


@pytest.mark.parametrize("qtype,K", [(syn.Q8_0, 256), (syn.Q8_0, 1024), (syn.Q4_K, 256), (syn.Q4_K, 768),
                                     (syn.Q5_K, 512), (syn.Q5_K, 1280), (syn.Q6_K, 2048)])
@pytest.mark.parametrize("N,M", [(128, 16), (200, 40), (384, 130), (130, 300)])
def test_fused_small(qtype, K, N, M):
    got, ref = _gemm(qtype, N, K, M)
    U.check_close(got, ref, "bf16", what=f"q{qtype} N{N} K{K} M{M}")


@pytest.mark.parametrize("N,M", [(128, 8), (256, 64), (200, 257)])
def test_fused_q6k_planes(N, M):
    got, ref = _gemm(syn.Q6_K, N, 2048, M, layout=1)
    U.check_close(got, ref, "bf16")


@pytest.mark.parametrize("ydt", ["f32", "f16"])
@pytest.mark.parametrize("qtype", [syn.Q5_K, syn.Q8_0])
def test_fused_out_dtypes(qtype, ydt):
    got, ref = _gemm(qtype, 256, 512, 48, ydt=ydt)
    U.check_close(got, ref, ydt, rel=2e-3)


def test_fused_f16_activations_no_residual():
    got, ref = _gemm(syn.Q4_K, 256, 512, 33, xdt="f16", residual=False)
    U.check_close(got, ref, "bf16")


def test_auto_path_picks_gemv_below_8_rows_and_fused_above():
    # same inputs through AUTO: M = 7 goes to the int8 GEMV (int8-path oracle),
    # M = 8 to the fused tensor-core GEMM (exact oracle)
    rs = syn.rng(3)
    N, K = 256, 1024
    w = syn.weight_blocks(rs, syn.Q5_K, N, K)
    for M in (7, 8):
        x = syn.normal(rs, (M, K), "bf16")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, syn.Q5_K, N, K, M)
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        g.gguf_mm_gemm(U.dev(w), syn.Q5_K, 0, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, None, y, g.GGUF_DT_F32,
                       ws, ws_bytes, g.GGUF_PATH_AUTO)
        torch.cuda.synchronize()
        if M == 7:
            ref = O.gemv_int8_path(w, syn.Q5_K, N, K, U.act_f32(x, "bf16"))
        else:
            ref = O.matmul_exact(U.act_f64(x, "bf16"), O.dequant(w, syn.Q5_K, N, K))
        U.check_close(U.host64(y), ref, "f32", rel=2e-3)


@pytest.mark.parametrize("qtype,layout", [(syn.Q6_K, 0), (syn.Q6_K, 1), (syn.Q5_K, 0)])
@pytest.mark.parametrize("M", [8, 512])
def test_fused_config_14336x4096(qtype, layout, M):
    # the prefill workload's shapes; rows sampled for the oracle
    rows = np.arange(0, M, max(1, M // 5))
    got, ref = _gemm(qtype, 14336, 4096, M, layout=layout, residual=False, seed=1002, rows=rows)
    U.check_close(got, ref, "bf16")


@pytest.mark.parametrize("M", [128, 512])
def test_fused_config_q8_0_2048x8192(M):
    rows = np.arange(0, M, max(1, M // 6))
    got, ref = _gemm(syn.Q8_0, 2048, 8192, M, residual=False, seed=1003, rows=rows)
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


def test_fused_split_k_residual_exact_and_deterministic():
    # 2 row tiles and K = 4096 leave most SMs idle, so the plan splits K; the
    # slices' sums meet in the workspace and the last slice adds them in a
    # fixed order: two runs agree bit for bit, and both match the oracle
    qtype, N, K, M = syn.Q4_K, 256, 4096, 40
    rs = syn.rng(4242)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    r = syn.normal(rs, (M, N), "bf16")
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qtype, N, K, M)
    assert ws_bytes > M * K * 2   # room for the partial tiles
    outs = []
    for fill in (0x00, 0xFF):   # stale workspace bytes (tickets included) must not matter
        ws = torch.full((ws_bytes,), fill, dtype=torch.uint8, device="cuda")
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        g.gguf_mm_gemm(U.dev(w), qtype, 0, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, U.dev(r, "bf16"), y,
                       g.GGUF_DT_BF16, ws, ws_bytes, g.GGUF_PATH_FUSED)
        torch.cuda.synchronize()
        assert g.gguf_mm_check_errors() == 0
        outs.append(U.host64(y))
    assert np.array_equal(outs[0], outs[1])
    ref = O.matmul_exact(U.act_f64(x, "bf16"), O.dequant(w, qtype, N, K), U.act_f64(r, "bf16"))
    U.check_close(outs[0], ref, "bf16")


def test_fused_tail_split_whole_then_halves():
    # 224 tiles on a 152-SM GB300: the plan keeps one round of 152 tiles whole
    # and splits the other 72 into K halves; stale workspace bytes must not
    # matter and two runs agree bit for bit
    qtype, N, K, M = syn.Q4_K, 14336, 1024, 512
    rs = syn.rng(4343)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    r = syn.normal(rs, (M, N), "bf16")
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qtype, N, K, M)
    outs = []
    for fill in (0x00, 0xFF):
        ws = torch.full((ws_bytes,), fill, dtype=torch.uint8, device="cuda")
        y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        g.gguf_mm_gemm(U.dev(w), qtype, 0, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, U.dev(r, "bf16"), y,
                       g.GGUF_DT_BF16, ws, ws_bytes, g.GGUF_PATH_FUSED)
        torch.cuda.synchronize()
        assert g.gguf_mm_check_errors() == 0
        outs.append(U.host64(y))
    assert np.array_equal(outs[0], outs[1])
    ref = O.matmul_exact(U.act_f64(x, "bf16"), O.dequant(w, qtype, N, K), U.act_f64(r, "bf16"))
    U.check_close(outs[0], ref, "bf16")
