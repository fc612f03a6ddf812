"""Calls issued back to back on one stream, with no synchronisation between
them: each kernel of a call may start (programmatic dependent launch) while the
previous call still runs, so this is where a race between a kernel's prologue
and its dependency wait would show.  Every call gets its own weights and its
own output; all are checked after one final synchronisation."""
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


# (qtype, layout, N, K, M): one-row tile kernel, pair kernel, direct kernel,
# bulk-copy kernel (raw Q6_K, Q8_0)
GEMV_CASES = [
    (syn.Q5_K, 0, 4096, 4096, 1),
    (syn.Q4_K, 0, 1000, 2048, 1),
    (syn.Q5_K, 0, 4096, 4096, 2),
    (syn.Q4_K, 0, 2000, 4096, 4),
    (syn.Q5_K, 0, 1000, 4096, 8),
    (syn.Q6_K, 1, 512, 2048, 2),
    (syn.Q6_K, 0, 512, 2048, 3),
    (syn.Q8_0, 0, 512, 2048, 1),
]


@pytest.mark.parametrize("qtype,layout,N,K,M", GEMV_CASES)
def test_gemv_back_to_back(qtype, layout, N, K, M):
    calls = 6
    rs = syn.rng(500 + qtype + M + N)
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, qtype, N, K, M)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")   # shared by all calls (same stream)
    ins = []
    for c in range(calls):
        w = syn.weight_blocks(rs, qtype, N, K)
        x = syn.normal(rs, (M, K), "bf16")
        r = syn.normal(rs, (M, N), "bf16")
        wd = U.dev(O.q6k_to_planes(w) if layout else w)
        ins.append((w, x, r, wd, U.dev(x, "bf16"), U.dev(r, "bf16"),
                    torch.empty((M, N), dtype=torch.bfloat16, device="cuda")))
    torch.cuda.synchronize()
    for w, x, r, wd, xd, rd, y in ins:
        g.gguf_mm_gemv(wd, qtype, layout, N, K, xd, g.GGUF_DT_BF16, M, rd, y, g.GGUF_DT_BF16, ws, ws_bytes)
    torch.cuda.synchronize()
    assert g.gguf_mm_check_errors() == 0
    for w, x, r, wd, xd, rd, y in ins:
        ref = O.gemv_int8_path(w, qtype, N, K, U.act_f32(x, "bf16"), U.act_f64(r, "bf16"))
        U.check_close(U.host64(y), ref, "bf16")


def test_gemv_chain_output_feeds_next_input():
    # y of call c is x of call c + 1 (N = K): each call must see its producer's
    # finished output, not a stale one
    qtype, N = syn.Q5_K, 2048
    rs = syn.rng(77)
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, qtype, N, N, 1)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    weights = [syn.weight_blocks(rs, qtype, N, N) for _ in range(4)]
    wds = [U.dev(w) for w in weights]
    x0 = syn.normal(rs, (1, N), "bf16")
    bufs = [U.dev(x0, "bf16")] + [torch.empty((1, N), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
    torch.cuda.synchronize()
    for c in range(4):
        g.gguf_mm_gemv(wds[c], qtype, 0, N, N, bufs[c], g.GGUF_DT_BF16, 1, None, bufs[c + 1], g.GGUF_DT_BF16,
                       ws, ws_bytes)
    torch.cuda.synchronize()
    assert g.gguf_mm_check_errors() == 0
    # check each call against the oracle applied to the input it actually read
    for c in range(4):
        xin = bufs[c].view(torch.int16).cpu().numpy().view(np.uint16)
        ref = O.gemv_int8_path(weights[c], qtype, N, N, O.bf16_bits_to_f32(xin))
        U.check_close(U.host64(bufs[c + 1]), ref, "bf16")


@pytest.mark.parametrize("qtype,layout,M", [(syn.Q5_K, 0, 96), (syn.Q6_K, 1, 40), (syn.Q8_0, 0, 300)])
def test_fused_gemm_back_to_back(qtype, layout, M):
    N, K, calls = 384, 2048, 4
    rs = syn.rng(600 + qtype + M)
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qtype, N, K, M)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ins = []
    for c in range(calls):
        w = syn.weight_blocks(rs, qtype, N, K)
        x = syn.normal(rs, (M, K), "bf16")
        wd = U.dev(O.q6k_to_planes(w) if layout else w)
        ins.append((w, x, wd, U.dev(x, "bf16"), torch.empty((M, N), dtype=torch.float32, device="cuda")))
    torch.cuda.synchronize()
    for w, x, wd, xd, y in ins:
        g.gguf_mm_gemm(wd, qtype, layout, N, K, xd, g.GGUF_DT_BF16, M, None, y, g.GGUF_DT_F32, ws, ws_bytes,
                       g.GGUF_PATH_FUSED)
    torch.cuda.synchronize()
    assert g.gguf_mm_check_errors() == 0
    for w, x, wd, xd, y in ins:
        ref = O.matmul_exact(U.act_f64(x, "bf16"), O.dequant(w, qtype, N, K))
        U.check_close(U.host64(y), ref, "f32", rel=2e-3)
