"""CPU checks of the C ABI: the library loads, exports every function that
include/gguf_mm.h declares, and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import gguf_quant_weight_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "gguf_mm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z_0-9]*\s*\*?\s*(gguf_[a-z0-9_]+)\s*\(", src,
                                 flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from gguf_quant_weight_gb300 import _build
    _build.build()
    return g.load_library()


def test_header_lists_the_entry_points():
    names = _declared()
    for n in ("gguf_mm_gemv", "gguf_mm_gemm", "gguf_mm_id", "gguf_mm_id_slots", "gguf_repack_q6k_planes",
              "gguf_dequant_padded",
              "gguf_dense_gemm", "gguf_mm_check_errors", "gguf_mm_workspace_size"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        assert name in g.exported_symbols(), f"binding lacks {name}"


def test_version_and_status_strings(lib):
    assert g.gguf_mm_version() >= 100
    assert g.status_string(0) == "ok"
    assert "aligned" in g.status_string(g.GGUF_ERR_MISALIGNED)


def test_argument_errors_need_no_gpu(lib):
    # null pointers / bad sizes / bad types are rejected before any CUDA call
    f = g.raw_status
    assert f("gguf_mm_gemv", None, 12, 0, 4, 256, None, 2, 1, None, None, 2, None, 0, None) == g.GGUF_ERR_INVALID_ARG
    assert f("gguf_mm_gemv", 16, 12, 0, 4, 100, 16, 2, 1, None, 16, 2, None, 0, None) == g.GGUF_ERR_INVALID_ARG
    assert f("gguf_mm_gemv", 16, 99, 0, 4, 256, 16, 2, 1, None, 16, 2, None, 0, None) == g.GGUF_ERR_UNSUPPORTED
    assert f("gguf_mm_gemv", 16, 12, 1, 4, 256, 16, 2, 1, None, 16, 2, None, 0, None) == g.GGUF_ERR_UNSUPPORTED
    assert f("gguf_mm_gemv", 18, 12, 0, 4, 256, 16, 2, 1, None, 16, 2, None, 0, None) == g.GGUF_ERR_MISALIGNED
    assert f("gguf_mm_gemv", 16, 12, 0, 4, 256, 16, 2, 1, None, 16, 2, None, 0, None) == g.GGUF_ERR_WORKSPACE
    assert f("gguf_mm_gemv", 16, 12, 0, 4, 256, 16, 2, 1, None, 16, 2, 16, 64, None) == g.GGUF_ERR_WORKSPACE
    assert f("gguf_mm_gemv", 16, 12, 0, 4, 256, 16, 2, 1, None, 16, 2, 24, 1024, None) == g.GGUF_ERR_MISALIGNED
    assert f("gguf_mm_gemm", 16, 12, 0, 4, 256, 16, 2, 8, None, 16, 2, None, 0, 9, None) == g.GGUF_ERR_INVALID_ARG
    assert f("gguf_repack_q6k_planes", 16, 16, 4, 0, None) == g.GGUF_ERR_INVALID_ARG
    assert f("gguf_dequant_padded", 16, 8, 0, 4, 64, 16, 2, 60, None) == g.GGUF_ERR_INVALID_ARG
    assert f("gguf_dense_gemm", 16, 1, 256, 4, 200, 16, 1, 8, None, 16, 2, None, 0, None) == g.GGUF_ERR_INVALID_ARG
    assert f("gguf_mm_id", 16, 12, 0, 4, 256, 16, 2, 8, None, 8, None, 16, 2, None, 0, None) == g.GGUF_ERR_INVALID_ARG
    # the MoE call with a chosen form: an unknown path value
    assert f("gguf_mm_id_path", 16, 12, 8, 256, 256, 16, 2, 1, 16, 2, 0, None, 16, 2, 16, 1 << 20, 7, None) == \
        g.GGUF_ERR_INVALID_ARG
    # the host-buffer GEMV: its own pointer rules, then the GEMV's, before any copy
    h = "gguf_mm_gemv_host"
    assert f(h, 16, 12, 0, 4, 256, None, 16, 2, 1, None, None, 32, 16, 2, 16, 4096, None) == g.GGUF_ERR_INVALID_ARG
    assert f(h, 16, 12, 0, 4, 256, 32, 16, 2, 1, None, None, None, 16, 2, 16, 4096, None) == g.GGUF_ERR_INVALID_ARG
    assert f(h, 16, 12, 0, 4, 256, 32, 16, 2, 1, 48, None, 32, 16, 2, 16, 4096, None) == g.GGUF_ERR_INVALID_ARG
    assert f(h, 16, 12, 0, 4, 256, 32, 18, 2, 1, None, None, 32, 16, 2, 16, 4096, None) == g.GGUF_ERR_MISALIGNED
    assert f(h, 16, 12, 0, 4, 256, 32, 16, 2, 1, None, None, 32, 16, 2, 16, 64, None) == g.GGUF_ERR_WORKSPACE


def test_workspace_sizes_are_consistent(lib):
    # GEMV: the quantized activation image, M rows of K codes with 16 pad bytes
    # after every 128, then 16 bytes per 32-value block and row, 256-rounded
    for M, K in ((1, 4096), (3, 768), (8, 14336), (2, 32)):
        img = M * (K + 16 * -(-K // 128)) + M * (K // 32) * 16
        assert g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, 13, 4096, K, M) == -(-img // 256) * 256
        assert g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, 13, 4096, K, M) >= -(-img // 256) * 256
    assert g.gguf_mm_workspace_size(g.GGUF_OP_GEMV, 13, 4096, 4096, 9) == 0
    assert g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, 13, 4096, 4096, 0) == 0


def test_per_slot_moe_rejects_bad_arguments_without_a_gpu(lib):
    f = g.raw_status
    assert f("gguf_mm_id_slots", 16, 12, 0, 4, 256, 16, 2, 8, None, 8, None, 16, 2, None, 0, None) == \
        g.GGUF_ERR_INVALID_ARG


def _r256(b):
    return -(-b // 256) * 256


def test_gemm_workspace_follows_the_tile_plan(lib):
    # (sized for 152 SMs when no device is current) activations in f16 and
    # their per-row f32 scales, then, when the plan splits K, one f32 [BN][128]
    # slot per slice of every split tile and one ticket per split tile
    act = lambda M, K: _r256(M * K * 2) + _r256(M * 4)
    # 2048 rows (16 row tiles) leave most SMs idle: every tile in 8 K slices at BN = 128
    assert g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, 8, 2048, 8192, 128) == \
        act(128, 8192) + _r256(16 * 8 * 128 * 128 * 4) + _r256(16 * 4)
    # 224 tiles at BN = 256: one round of 152 whole tiles, the other 72 in K halves
    assert g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, 13, 14336, 4096, 512) == \
        act(512, 4096) + _r256(72 * 2 * 256 * 128 * 4) + _r256(72 * 4)
    # 896 tiles: whole rounds only, no split
    assert g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, 13, 14336, 4096, 2048) == act(2048, 4096)


def test_moe_form_rule(lib, monkeypatch):
    # the decode form up to a per-format number of routed rows (T * top_k), as
    # the header states, and the routed tensor-core path above it; the tests'
    # mirror of the rule agrees; GGUF_MM_MOE_MV=0 keeps every batch routed
    from tests import gpu_util as U
    limits = {12: 128, 13: 128, 10: 128, 11: 128, 14: 128, 8: 16, 2: 32, 3: 32, 6: 32, 7: 32}
    for qt, lim in limits.items():
        assert U.moe_mv_max_rows(qt) == lim
        for top_k in (1, 2, 8):
            for T in sorted({1, max(1, lim // top_k), lim // top_k + 1, 4 * lim}):
                want = g.GGUF_PATH_GEMV if T * top_k <= lim else g.GGUF_PATH_FUSED
                assert g.gguf_mm_id_form(qt, T, top_k) == want, (qt, T, top_k)
    assert g.gguf_mm_id_form(99, 1, 1) == g.GGUF_ERR_INVALID_ARG
    assert g.gguf_mm_id_form(12, 0, 8) == g.GGUF_ERR_INVALID_ARG
    assert g.gguf_mm_id_form(12, 1, 0) == g.GGUF_ERR_INVALID_ARG
    monkeypatch.setenv("GGUF_MM_MOE_MV", "0")
    assert g.gguf_mm_id_form(12, 1, 8) == g.GGUF_PATH_FUSED


def test_auto_path_table(lib):
    # the measured crossovers, by format and shape class (up to 8192 weight rows / more)
    big, small = (14336, 4096), (4096, 4096)
    want = {(12, 0): (9, 7), (13, 0): (9, 6), (14, 1): (7, 4), (14, 0): (3, 2), (8, 0): (6, 2),
            (2, 0): (6, 2), (3, 0): (6, 3), (6, 0): (6, 3), (7, 0): (5, 2), (10, 0): (4, 2), (11, 0): (5, 4)}
    for (qt, lay), (c_small, c_big) in want.items():
        for (n, k), c in ((small, c_small), (big, c_big)):
            first_fused = next(M for M in range(1, 12)
                               if g.gguf_mm_auto_path(qt, lay, n, k, M, g.GGUF_DT_BF16) == g.GGUF_PATH_FUSED)
            assert first_fused == min(c, 9), (qt, lay, n, k)
