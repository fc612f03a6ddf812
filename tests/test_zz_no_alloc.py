"""gguf_dense_gemm_noalloc: the dense GEMM for callers that may not obtain
device memory (their host program owns every allocation, or a cudaMalloc would
synchronize the device at the wrong moment).  It keeps its scratch in an array
built into the library instead of a caller workspace.

Checked here through the C ABI: two calls in a row (different activations each
time, so the shared array is reused) against the workspace entry point
gguf_dense_gemm on the same inputs, within the bf16-output bound the other GEMM
tests use; and the size limit is refused before anything runs.  This file is
collected last so that, when it fails, a run that stops at the first failure
has already run every other test."""
import numpy as np
import pytest
import torch

import gguf_quant_weight_gb300 as g
import gguf_synth as syn
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


def _decoded_weight(N, K, seed):
    w = syn.weight_blocks(syn.rng(seed), syn.Q8_0, N, K)
    ld = K + 64
    wd = torch.empty((N, ld), dtype=torch.float16, device="cuda")
    g.gguf_dequant_padded(U.dev(w), syn.Q8_0, 0, N, K, wd, g.GGUF_DT_F16, ld)
    return wd, ld


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    N, K, M = 384, 1024, 200
    wd, ld = _decoded_weight(N, K, 5)
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_DENSE, 0, N, K, M)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    for call in range(2):
        rs = syn.rng(100 + call)
        x = U.dev(syn.normal(rs, (M, K), "bf16"), "bf16")
        r = U.dev(syn.normal(rs, (M, N), "bf16"), "bf16")
        ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        got = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        g.gguf_dense_gemm(wd, g.GGUF_DT_F16, ld, N, K, x, g.GGUF_DT_BF16, M, r, ref, g.GGUF_DT_BF16, ws, ws_bytes)
        g.gguf_dense_gemm_noalloc(wd, g.GGUF_DT_F16, ld, N, K, x, g.GGUF_DT_BF16, M, r, got, g.GGUF_DT_BF16)
        torch.cuda.synchronize()
        U.check_close(U.host64(got), U.host64(ref), "bf16", what=f"call {call}")
    assert g.gguf_mm_check_errors() == 0


def test_noalloc_refuses_problems_beyond_its_scratch():
    # M * K * 2 bytes above 8 MiB: rejected on the host, nothing launched
    N, K, M = 128, 8192, 1024
    wd, ld = _decoded_weight(N, K, 6)
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GGUFError) as e:
        g.gguf_dense_gemm_noalloc(wd, g.GGUF_DT_F16, ld, N, K, x, g.GGUF_DT_BF16, M, None, y, g.GGUF_DT_BF16)
    assert e.value.status == g.GGUF_ERR_WORKSPACE
    assert torch.count_nonzero(y).item() == 0
