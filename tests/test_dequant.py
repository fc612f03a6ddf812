"""Decode-once K-padded buffer: every value is the exact decoded weight
correctly rounded to f16/bf16 (bit for bit against the oracle's RN(w)), pad
columns are zero, and padding changes only the stride (ROCm llama.cpp PR #37
"one-time K-padded f16 dequantization for prefill GEMMs", "How it works" and
"Correctness")."""
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


def _decode(w, qtype, N, K, ld, odt, layout=0):
    out = U.guarded((N, ld), torch.int16, fill=0x7777)
    g.gguf_dequant_padded(U.dev(w), qtype, layout, N, K, out.t, U.DT[odt], ld)
    torch.cuda.synchronize()
    out.check("decoded buffer")
    return out.t.cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("qtype", [syn.Q4_0, syn.Q4_1, syn.Q5_0, syn.Q5_1, syn.Q8_0, syn.Q2_K, syn.Q3_K, syn.Q4_K,
                                   syn.Q5_K, syn.Q6_K])
@pytest.mark.parametrize("odt", ["f16", "bf16"])
@pytest.mark.parametrize("N,K,pad", [(3, 256, 64), (65, 512, 0), (17, 1024, 64)])
def test_dequant_padded(qtype, odt, N, K, pad):
    rs = syn.rng(qtype * 100 + N + K)
    w = syn.weight_blocks(rs, qtype, N, K)
    ld = K + pad
    bits = _decode(w, qtype, N, K, ld, odt)
    assert np.array_equal(bits, O.dequant_padded_bits(w, qtype, N, K, ld, odt))   # pad columns included


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K])
@pytest.mark.parametrize("odt", ["f16", "bf16"])
def test_dequant_kquant_min_rounded_once(qtype, odt):
    # d*sc*q and dmin*m close to each other, so that their difference needs
    # more bits than the output type holds: one rounding of the exact weight,
    # never the f32 difference rounded again
    N, K = 64, 512
    rs = syn.rng(31 + qtype)
    w = syn.weight_blocks(rs, qtype, N, K).reshape(-1, 144 if qtype == syn.Q4_K else 176)
    w[:, 0:2] = np.frombuffer(np.float16(0.0123).tobytes(), np.uint8)
    w[:, 2:4] = np.frombuffer(np.float16(0.0119).tobytes(), np.uint8)
    w = w.reshape(N, -1)
    bits = _decode(w, qtype, N, K, K, odt)
    assert np.array_equal(bits, O.dequant_padded_bits(w, qtype, N, K, K, odt))


def test_dequant_planes_equals_blocks():
    N, K = 40, 1024
    rs = syn.rng(77)
    w = syn.weight_blocks(rs, syn.Q6_K, N, K)
    a = torch.empty((N, K + 64), dtype=torch.int16, device="cuda")
    b = torch.empty((N, K + 64), dtype=torch.int16, device="cuda")
    g.gguf_dequant_padded(U.dev(w), syn.Q6_K, 0, N, K, a, g.GGUF_DT_F16, K + 64)
    g.gguf_dequant_padded(U.dev(O.q6k_to_planes(w)), syn.Q6_K, 1, N, K, b, g.GGUF_DT_F16, K + 64)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_dequant_config_q8_0_2048x8192_padded():
    N, K = 2048, 8192
    rs = syn.rng(1003)
    w = syn.weight_blocks(rs, syn.Q8_0, N, K)
    out = torch.empty((N, K + 64), dtype=torch.int16, device="cuda")
    g.gguf_dequant_padded(U.dev(w), syn.Q8_0, 0, N, K, out, g.GGUF_DT_BF16, K + 64)
    torch.cuda.synchronize()
    bits = out.cpu().numpy().view(np.uint16)
    rows = np.arange(0, N, 97)
    ref = O.dequant_padded_bits(w[rows], syn.Q8_0, len(rows), K, K + 64, "bf16")
    assert np.array_equal(bits[rows], ref)
