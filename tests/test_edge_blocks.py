"""The method's edge blocks on every GPU path: hand-built weight tensors whose
blocks hit the ends of each field (GGUF Support Proposal for mobius, 7.3 / 7.4
block structs; OpenVINO PR #39119 "Transformation" for the Q6_K fields):

  allff      every quant and scale byte 0xFF, d = dmin = 1 (Q4_K 882, Q5_K 1890,
             Q6_K -31, Q8_0 -1, Q4_0 7, Q4_1 16, Q5_0 15, Q5_1 32, Q2_K 30,
             Q3_K 93 per the oracle's invariants)
  zero       every byte 0 (d = 0: all weights zero)
  extreme    Q8_0 q = -128 everywhere; K-quants: every 6-bit scale and min 63;
             Q6_K: every scale -128 or 127; Q4_0/Q4_1/Q5_0/Q5_1: codes 0 and
             15 (31 with every fifth bit set); Q2_K: every scale and min 15;
             Q3_K: 6-bit scales 0 or 63 with every 2-bit code 0
  half_d0    random blocks, d (and dmin) = 0 in every other block
  tiny_d     random blocks with d, dmin = |N(0,1)| * 1e-7 (f16 subnormals)
  q6_scales  random blocks, Q6_K scales uniform over the whole i8 range
  nan_d      random blocks, one block of weight row 5 with d = NaN: that
             row's outputs are NaN and no other output is

Outputs are f32, so the bounds hold raw: 1e-4 * max|ref| on the int8 GEMV
path against the int8-path oracle, 2e-3 * max|ref| on the f16 tensor-core
paths against the exact oracle; NaN must appear exactly where the oracle has
it.  The decode-once buffer is compared bit for bit (NaN by position)."""
import numpy as np
import pytest
import torch

import gguf_quant_weight_gb300 as g
import gguf_synth as syn
from oracle import gguf_oracle as O
from tests import gpu_util as U

pytestmark = pytest.mark.gpu

QTYPES = [syn.Q8_0, syn.Q4_K, syn.Q5_K, syn.Q6_K, syn.Q4_0, syn.Q4_1, syn.Q5_0, syn.Q5_1, syn.Q2_K, syn.Q3_K]
PATTERNS = ["allff", "zero", "extreme", "half_d0", "tiny_d", "q6_scales", "nan_d"]
N, K = 128, 2048
F16_ONE = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)
F16_NAN = np.array([0x00, 0x7E], np.uint8)


def _d_fields(qtype):
    """Byte offsets of the f16 scale fields d (and dmin) inside a block."""
    return {syn.Q8_0: [0], syn.Q4_K: [0, 2], syn.Q5_K: [0, 2], syn.Q6_K: [208], syn.Q4_0: [0], syn.Q5_0: [0],
            syn.Q4_1: [0, 2], syn.Q5_1: [0, 2], syn.Q2_K: [80, 82], syn.Q3_K: [108]}[qtype]


def edge_weights(qtype, pattern, seed=0):
    rs = syn.rng(700 + 13 * qtype + PATTERNS.index(pattern) + seed)
    bb = syn.BLOCK_BYTES[qtype]
    w = syn.weight_blocks(rs, qtype, N, K).reshape(-1, bb)
    nb = w.shape[0]
    if pattern == "allff":
        w[:] = 0xFF
        for o in _d_fields(qtype):
            w[:, o:o + 2] = F16_ONE
    elif pattern == "zero":
        w[:] = 0
    elif pattern == "extreme":
        if qtype == syn.Q8_0:
            w[:, 2:34] = 0x80                       # q = -128
        elif qtype in (syn.Q4_K, syn.Q5_K):
            w[:, 4:16] = 0xFF                       # every 6-bit scale and min = 63
        elif qtype == syn.Q6_K:
            w[:, 192:208] = np.where(rs.integers(0, 2, (nb, 16)) > 0, 0x7F, 0x80).astype(np.uint8)
        elif qtype == syn.Q2_K:                     # every scale and min 15
            w[:, 0:16] = 0xFF
        elif qtype == syn.Q3_K:                     # every 6-bit scale 63 or 0 (w scale 31 or -32), codes 0
            w[:, 96:108] = np.where(rs.integers(0, 2, (nb, 12)) > 0, 0xFF, 0x00).astype(np.uint8)
            w[:, 32:96] = 0
        else:                                       # 32-value blocks: codes 0 and 15 (31), every fifth bit set
            qo = {syn.Q4_0: 2, syn.Q4_1: 4, syn.Q5_0: 6, syn.Q5_1: 8}[qtype]
            w[:, qo:qo + 16] = np.where(rs.integers(0, 2, (nb, 16)) > 0, 0x0F, 0xF0).astype(np.uint8)
            if qtype in (syn.Q5_0, syn.Q5_1):
                w[:, qo - 4:qo] = 0xFF
    elif pattern == "half_d0":
        for o in _d_fields(qtype):
            w[::2, o:o + 2] = 0
    elif pattern == "tiny_d":
        for o in _d_fields(qtype):
            v = (np.abs(rs.standard_normal(nb)) * 1e-7).astype(np.float16)
            w[:, o:o + 2] = v.view(np.uint8).reshape(nb, 2)
    elif pattern == "q6_scales":
        if qtype == syn.Q6_K:
            w[:, 192:208] = rs.integers(0, 256, (nb, 16), dtype=np.uint8)
    elif pattern == "nan_d":
        per_row = nb // N
        w[5 * per_row + per_row // 2, _d_fields(qtype)[0]:_d_fields(qtype)[0] + 2] = F16_NAN
    return np.ascontiguousarray(w.reshape(N, -1))


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


def _x(M, seed=1):
    return syn.normal(syn.rng(seed + M), (M, K), "bf16")


@pytest.mark.parametrize("pattern", PATTERNS)
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("M", [1, 3])
def test_edge_blocks_gemv(qtype, pattern, M):
    w = edge_weights(qtype, pattern)
    x = _x(M)
    y = U.guarded((M, N), torch.float32)
    nws = g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, qtype, N, K, M)
    ws = U.workspace(nws)
    g.gguf_mm_gemv(U.dev(w), qtype, 0, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, None, y.t, g.GGUF_DT_F32, ws.t,
                   nws)
    torch.cuda.synchronize()
    y.check("y")
    assert g.gguf_mm_check_errors() == 0
    with np.errstate(invalid="ignore"):
        ref = O.gemv_int8_path(w, qtype, N, K, U.act_f32(x, "bf16"))
    got = U.host64(y.t)
    if pattern == "zero":
        assert np.all(got == 0)
    U.check_close(got, ref, "f32", allow_nan=True, what=f"{pattern} q{qtype} M{M}")


@pytest.mark.parametrize("pattern", PATTERNS)
@pytest.mark.parametrize("qtype", QTYPES)
def test_edge_blocks_fused(qtype, pattern):
    M = 40
    w = edge_weights(qtype, pattern)
    x = _x(M)
    y = U.guarded((M, N), torch.float32)
    nws = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qtype, N, K, M)
    ws = U.workspace(nws)
    g.gguf_mm_gemm(U.dev(w), qtype, 0, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, None, y.t, g.GGUF_DT_F32, ws.t,
                   nws, g.GGUF_PATH_FUSED)
    torch.cuda.synchronize()
    y.check("y")
    ws.check("workspace")
    assert g.gguf_mm_check_errors() == 0
    with np.errstate(invalid="ignore"):
        ref = O.matmul_exact(U.act_f64(x, "bf16"), O.dequant(w, qtype, N, K))
    U.check_close(U.host64(y.t), ref, "f32", rel=2e-3, allow_nan=True, what=f"{pattern} q{qtype}")


@pytest.mark.parametrize("pattern", PATTERNS)
@pytest.mark.parametrize("qtype", QTYPES)
@pytest.mark.parametrize("odt", ["f16", "bf16"])
def test_edge_blocks_decode_once_and_dense(qtype, pattern, odt):
    w = edge_weights(qtype, pattern)
    ld = K + 64
    out = U.guarded((N, ld), torch.int16, fill=0x1111)
    g.gguf_dequant_padded(U.dev(w), qtype, 0, N, K, out.t, U.DT[odt], ld)
    torch.cuda.synchronize()
    out.check("decoded")
    bits = out.t.cpu().numpy().view(np.uint16)
    with np.errstate(invalid="ignore"):
        ref = O.dequant_padded_bits(w, qtype, N, K, ld, odt)
    vals = bits.view(np.float16).astype(np.float64) if odt == "f16" else O.bf16_bits_to_f64(bits)
    rvals = ref.view(np.float16).astype(np.float64) if odt == "f16" else O.bf16_bits_to_f64(ref)
    nan = np.isnan(rvals)
    assert np.array_equal(np.isnan(vals), nan)
    assert np.array_equal(bits[~nan], ref[~nan])
    # the dense GEMM on that buffer (f32 out), against the product with the rounded weights
    M = 24
    x = _x(M)
    y = U.guarded((M, N), torch.float32)
    nws = g.gguf_mm_workspace_size(g.GGUF_OP_DENSE, 0, N, K, M)
    ws = U.workspace(nws)
    g.gguf_dense_gemm(out.t, U.DT[odt], ld, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, None, y.t, g.GGUF_DT_F32,
                      ws.t, nws)
    torch.cuda.synchronize()
    y.check("y")
    assert g.gguf_mm_check_errors() == 0
    with np.errstate(invalid="ignore"):
        ref_y = O.matmul_exact(U.act_f64(x, "bf16"), rvals[:, :K])
    U.check_close(U.host64(y.t), ref_y, "f32", rel=2e-3, allow_nan=True, what=f"{pattern} q{qtype} {odt}")


@pytest.mark.parametrize("T,top_k", [(6, 2), (80, 2)])
@pytest.mark.parametrize("qtype", QTYPES)
def test_edge_blocks_moe(qtype, T, top_k):
    # every pattern is one expert; T * top_k = 12 rows take the decode form
    # (every format), 160 rows the routed tensor-core path
    E = len(PATTERNS)
    wE = np.concatenate([edge_weights(qtype, p) for p in PATTERNS])
    x = syn.normal(syn.rng(T), (T, K), "bf16")
    ids = np.stack([syn.rng(100 * T + t).choice(E, size=top_k, replace=False) for t in range(T)]).astype(np.int32)
    ids[0, 0] = PATTERNS.index("nan_d")
    y = U.guarded((T, top_k, N), torch.float32)
    nws = g.gguf_mm_workspace_size(g.GGUF_OP_ID, qtype, N, K, T, E, top_k)
    ws = U.workspace(nws)
    g.gguf_mm_id(U.dev(wE), qtype, E, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, T, U.dev(ids), top_k, None, y.t,
                 g.GGUF_DT_F32, ws.t, nws)
    torch.cuda.synchronize()
    y.check("y")
    ws.check("workspace")
    assert g.gguf_mm_check_errors() == 0
    decode_form = U.moe_decode_form(qtype, T * top_k)
    with np.errstate(invalid="ignore"):
        if decode_form:
            ref = O.moe_mv_id_int8(wE, qtype, E, N, K, U.act_f32(x, "bf16"), ids)
        else:
            ref = O.moe_mm_id_exact(wE, qtype, E, N, K, U.act_f64(x, "bf16"), ids)
    got = U.host64(y.t)
    for e, p in enumerate(PATTERNS):   # each expert against its own scale
        sel = ids == e
        if sel.any():
            U.check_close(got[sel], ref[sel], "f32", rel=1e-4 if decode_form else 2e-3, allow_nan=True,
                          what=f"expert {p}")
