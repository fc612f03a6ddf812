"""Q6_K plane regrouping on the GPU: bit-exact against the oracle, round trip,
partial last tile."""
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


@pytest.mark.parametrize("nblk", [1, 63, 64, 65, 200, 1024 + 17])
def test_repack_bit_exact_and_roundtrip(nblk):
    rs = syn.rng(nblk)
    w = syn.weight_blocks(rs, syn.Q6_K, nblk, 256)
    src = U.dev(w)
    planes = torch.full((w.size,), 0xAB, dtype=torch.uint8, device="cuda")
    back = torch.full((w.size,), 0xCD, dtype=torch.uint8, device="cuda")
    g.gguf_repack_q6k_planes(src, planes, nblk, 0)
    g.gguf_repack_q6k_planes(planes, back, nblk, 1)
    torch.cuda.synchronize()
    assert np.array_equal(planes.cpu().numpy(), O.q6k_to_planes(w))
    assert np.array_equal(back.cpu().numpy().reshape(w.shape), w)


def test_repack_config_14336x4096():
    # the prefill workload's Q6_K tensor: 229,376 blocks, 48,168,960 bytes
    N, K = 14336, 4096
    nblk = N * K // 256
    rs = syn.rng(1002)
    w = syn.weight_blocks(rs, syn.Q6_K, N, K)
    planes = torch.empty(w.size, dtype=torch.uint8, device="cuda")
    g.gguf_repack_q6k_planes(U.dev(w), planes, nblk, 0)
    torch.cuda.synchronize()
    assert w.size == 48_168_960
    assert np.array_equal(planes.cpu().numpy(), O.q6k_to_planes(w))


def test_repack_rejects_overlap():
    buf = torch.empty(210 * 4, dtype=torch.uint8, device="cuda")
    with pytest.raises(g.GGUFError):
        g.gguf_repack_q6k_planes(buf, buf, 4, 0)
