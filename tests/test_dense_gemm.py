"""Decode-once arm: K-padded decoded buffer + our own dense tcgen05 GEMM,
against the exact f64 oracle (ROCm llama.cpp PR #37, "How it works")."""
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


def _dense(qtype, N, K, M, wdt="f16", ydt="bf16", residual=True, seed=0):
    rs = syn.rng(seed + N + 3 * K + 7 * M + qtype)
    w = syn.weight_blocks(rs, qtype, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    r = syn.normal(rs, (M, N), ydt) if residual else None
    ld = K + 64
    wd = torch.empty((N, ld), dtype=U.TORCH_DT[wdt], device="cuda")
    g.gguf_dequant_padded(U.dev(w), qtype, 0, N, K, wd, U.DT[wdt], ld)
    y = torch.empty((M, N), dtype=U.TORCH_DT[ydt], device="cuda")
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_DENSE, 0, N, K, M)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    g.gguf_dense_gemm(wd, U.DT[wdt], ld, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M,
                      None if r is None else U.dev(r, ydt), y, U.DT[ydt], ws, ws_bytes)
    torch.cuda.synchronize()
    ref = O.matmul_exact(U.act_f64(x, "bf16"), O.dequant(w, qtype, N, K), None if r is None else U.act_f64(r, ydt))
    return U.host64(y), ref


@pytest.mark.parametrize("N,K,M", [(128, 256, 16), (200, 512, 33), (256, 1024, 300), (130, 768, 1),
                                   (384, 512, 257), (1000, 256, 64)])
@pytest.mark.parametrize("qtype", [syn.Q8_0, syn.Q4_K])
def test_dense_gemm_f16(qtype, N, K, M):
    got, ref = _dense(qtype, N, K, M)
    U.check_close(got, ref, "bf16")


@pytest.mark.parametrize("ydt", ["f32", "f16"])
def test_dense_gemm_out_dtypes(ydt):
    got, ref = _dense(syn.Q5_K, 256, 512, 48, ydt=ydt)
    U.check_close(got, ref, ydt, rel=2e-3)


def test_dense_gemm_bf16_weights_reported():
    # bf16 decoded weights carry 8 significant bits: the error is reported and
    # gated at twice the f16 bound (the bf16 arm of the decode-once comparison)
    got, ref = _dense(syn.Q8_0, 512, 2048, 128, wdt="bf16")
    rel = U.check_close(got, ref, "bf16", rel=4e-3)
    print(f"bf16 decode-once error: {rel:.2e} of max|ref|")


def test_dense_gemm_config_q8_0_2048x8192_m512():
    N, K, M = 2048, 8192, 512
    rs = syn.rng(1003)
    w = syn.weight_blocks(rs, syn.Q8_0, N, K)
    x = syn.normal(rs, (M, K), "bf16")
    ld = K + 64
    wd = torch.empty((N, ld), dtype=torch.float16, device="cuda")
    g.gguf_dequant_padded(U.dev(w), syn.Q8_0, 0, N, K, wd, g.GGUF_DT_F16, ld)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_DENSE, 0, N, K, M)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    g.gguf_dense_gemm(wd, g.GGUF_DT_F16, ld, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, None, y, g.GGUF_DT_BF16,
                      ws, ws_bytes)
    torch.cuda.synchronize()
    rows = np.arange(0, M, 61)
    ref = O.matmul_exact(U.act_f64(x[rows], "bf16"), O.dequant(w, syn.Q8_0, N, K))
    U.check_close(U.host64(y)[rows], ref, "bf16")
    assert g.gguf_mm_check_errors() == 0
