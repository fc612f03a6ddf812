"""Decode-once K-padded buffer: every value is the exact decoded weight rounded
to f16/bf16 (one of its two neighbours in the output type: the kernel computes
the K-quant value in f32 first), pad columns are zero, and padding changes only
the stride."""
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


def _bits_to_f64(bits, odt):
    if odt == "f16":
        return bits.view(np.float16).astype(np.float64)
    return O.bf16_bits_to_f64(bits)


def _faithful(got_bits, w64, odt):
    """got is RN(w) exactly, or one of the two output-type neighbours of w."""
    got = _bits_to_f64(got_bits, odt)
    rn = _bits_to_f64(O.round_f64_to_f16_bits(w64) if odt == "f16" else O.round_f64_to_bf16_bits(w64), odt)
    exact_match = np.mean(got == rn)
    ulp = 2 * U.half_ulp(w64, odt)
    assert np.all(np.abs(got - w64) <= ulp * (1 + 1e-9) + 2.0 ** -24), "not faithfully rounded"
    return exact_match


@pytest.mark.parametrize("qtype", [syn.Q8_0, syn.Q4_K, syn.Q5_K, syn.Q6_K])
@pytest.mark.parametrize("odt", ["f16", "bf16"])
@pytest.mark.parametrize("N,K,pad", [(3, 256, 64), (65, 512, 0), (17, 1024, 64)])
def test_dequant_padded(qtype, odt, N, K, pad):
    rs = syn.rng(qtype * 100 + N + K)
    w = syn.weight_blocks(rs, qtype, N, K)
    ld = K + pad
    out = torch.full((N, ld), 0x7777, dtype=torch.int16, device="cuda")
    g.gguf_dequant_padded(U.dev(w), qtype, 0, N, K, out, U.DT[odt], ld)
    torch.cuda.synchronize()
    bits = out.cpu().numpy().view(np.uint16)
    assert np.all(bits[:, K:] == 0)
    match = _faithful(bits[:, :K], O.dequant(w, qtype, N, K), odt)
    assert match > 0.999
    if qtype in (syn.Q8_0, syn.Q6_K):   # products exact in f32: correctly rounded
        assert match == 1.0


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
