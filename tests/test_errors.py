"""Error reporting on the GPU: argument checks return before launching, and a
bounded device wait that expires is reported through the status word (no GPU
fault is involved: the probe waits on a barrier nothing completes)."""
import pytest
import torch

import gguf_quant_weight_gb300 as g
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    U.require_gpu()


def test_bounded_wait_reports_timeout_and_clears():
    assert g.gguf_mm_check_errors() == 0
    g.gguf_mm_debug_timeout(1000)
    assert g.gguf_mm_check_errors() == g.GGUF_ERR_TIMEOUT
    assert g.gguf_mm_check_errors() == 0          # cleared by the read


def test_misaligned_pointer_rejected():
    w = torch.zeros(144 * 4 + 16, dtype=torch.uint8, device="cuda")
    x = torch.zeros((1, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((1, 4), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GGUFError) as e:
        g.gguf_mm_gemv(w.data_ptr() + 2, g.GGUF_Q4_K, 0, 4, 256, x, g.GGUF_DT_BF16, 1, None, y, g.GGUF_DT_BF16,
                       *U.gemv_workspace(1, 256))
    assert e.value.status == g.GGUF_ERR_MISALIGNED
    ws, n = U.gemv_workspace(1, 256)
    with pytest.raises(g.GGUFError) as e:
        g.gguf_mm_gemv(w, g.GGUF_Q4_K, 0, 4, 256, x, g.GGUF_DT_BF16, 1, None, y, g.GGUF_DT_BF16,
                       ws.data_ptr() + 8, n)
    assert e.value.status == g.GGUF_ERR_MISALIGNED


def test_gemv_workspace_required():
    w = torch.zeros(144 * 4, dtype=torch.uint8, device="cuda")
    x = torch.zeros((2, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((2, 4), dtype=torch.bfloat16, device="cuda")
    ws, n = U.gemv_workspace(2, 256)
    for buf, size in ((None, 0), (ws, n - 16)):
        with pytest.raises(g.GGUFError) as e:
            g.gguf_mm_gemv(w, g.GGUF_Q4_K, 0, 4, 256, x, g.GGUF_DT_BF16, 2, None, y, g.GGUF_DT_BF16, buf, size)
        assert e.value.status == g.GGUF_ERR_WORKSPACE


def test_gemv_rejects_too_many_rows():
    w = torch.zeros(144 * 4, dtype=torch.uint8, device="cuda")
    x = torch.zeros((9, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((9, 4), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.GGUFError) as e:
        g.gguf_mm_gemv(w, g.GGUF_Q4_K, 0, 4, 256, x, g.GGUF_DT_BF16, 9, None, y, g.GGUF_DT_BF16,
                       *U.gemv_workspace(8, 256))
    assert e.value.status == g.GGUF_ERR_UNSUPPORTED
