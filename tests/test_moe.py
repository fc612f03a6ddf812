"""MoE expert GEMM (gguf_mm_id) against the exact oracle (llama.cpp PR #28301,
"Overview": every routed (token, slot) row multiplies its expert's weight)."""
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


def _run(qtype, E, N, K, T, top_k, ids, residual=False, ydt="bf16", seed=0, token_rows=None, sentinel=None):
    rs = syn.rng(seed + E + N + K + T)
    wE = syn.weight_blocks(rs, qtype, E * N, K)
    x = syn.normal(rs, (T, K), "bf16")
    r = syn.normal(rs, (T, top_k, N), ydt) if residual else None
    yb = U.guarded((T, top_k, N), U.TORCH_DT[ydt], fill=float("nan") if sentinel is None else sentinel)
    y = yb.t
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_ID, qtype, N, K, T, E, top_k)
    ws = U.workspace(ws_bytes, 0x6B)
    g.gguf_mm_id(U.dev(wE), qtype, E, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, T, U.dev(ids.astype(np.int32)),
                 top_k, None if r is None else U.dev(r, ydt), y, U.DT[ydt], ws.t, ws_bytes)
    torch.cuda.synchronize()
    yb.check("y")
    ws.check("workspace")
    assert g.gguf_mm_check_errors() == 0
    rr = None if r is None else U.act_f64(r, ydt)
    if mv_form(qtype, T * top_k):
        ref = O.moe_mv_id_int8(wE, qtype, E, N, K, U.act_f32(x, "bf16"), ids, rr)
    else:
        ref = O.moe_mm_id_exact(wE, qtype, E, N, K, U.act_f64(x, "bf16"), ids, rr, token_rows=token_rows)
    return U.host64(y), ref


def mv_form(qtype, entries):
    # the library's decode form: up to a per-format number of routed rows are
    # computed one int8 GEMV per row (the GEMV's arithmetic)
    return U.moe_decode_form(qtype, entries)


def _distinct_ids(rs, T, E, top_k):
    return np.stack([rs.choice(E, size=top_k, replace=False) for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,top_k", [(1, 1), (5, 2), (40, 4), (130, 2)])
@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K, syn.Q8_0])
def test_moe_small_all_rows(qtype, T, top_k):
    E, N, K = 8, 256, 512
    ids = _distinct_ids(syn.rng(T + top_k), T, E, top_k)
    got, ref = _run(qtype, E, N, K, T, top_k, ids)
    U.check_close(got.reshape(T * top_k, N), ref.reshape(T * top_k, N), "bf16")


@pytest.mark.parametrize("qtype", [syn.Q4_0, syn.Q4_1, syn.Q5_0, syn.Q5_1, syn.Q2_K, syn.Q3_K])
def test_moe_32_value_formats(qtype):
    # the routed tensor-core path (T * top_k > 128 rows); also Q2_K / Q3_K (K % 2048)
    E, N, K, T, top_k = 6, 128, 512 if syn.BLOCK_VALUES[qtype] == 32 else 2048, 70, 2
    ids = _distinct_ids(syn.rng(qtype), T, E, top_k)
    got, ref = _run(qtype, E, N, K, T, top_k, ids)
    U.check_close(got.reshape(-1, N), ref.reshape(-1, N), "bf16")


def test_moe_q6k():
    E, N, K, T, top_k = 4, 128, 2048, 24, 2
    ids = _distinct_ids(syn.rng(9), T, E, top_k)
    got, ref = _run(syn.Q6_K, E, N, K, T, top_k, ids)
    U.check_close(got.reshape(-1, N), ref.reshape(-1, N), "bf16")


def test_moe_one_expert_spans_several_tiles_with_residual():
    # 300 rows on one expert: work items of 128, 128 and 44 rows
    E, N, K, T, top_k = 4, 384, 256, 300, 1
    ids = np.full((T, 1), 2, np.int32)
    got, ref = _run(syn.Q4_K, E, N, K, T, top_k, ids, residual=True)
    U.check_close(got.reshape(-1, N), ref.reshape(-1, N), "bf16")


def test_moe_invalid_ids_leave_rows_untouched():
    E, N, K, T, top_k = 8, 128, 256, 10, 2
    ids = _distinct_ids(syn.rng(3), T, E, top_k)
    ids[2, 1] = -1
    ids[7, 0] = E
    got, ref = _run(syn.Q4_K, E, N, K, T, top_k, ids, sentinel=1024.0)
    valid = (ids >= 0) & (ids < E)
    assert np.all(got[~valid] == 1024.0)
    U.check_close(got[valid], ref[valid], "bf16")


def test_moe_f32_output():
    E, N, K, T, top_k = 8, 256, 512, 17, 3
    ids = _distinct_ids(syn.rng(4), T, E, top_k)
    got, ref = _run(syn.Q5_K, E, N, K, T, top_k, ids, ydt="f32")
    U.check_close(got.reshape(-1, N), ref.reshape(-1, N), "f32", rel=2e-3)


@pytest.mark.parametrize("T", [32, 64, 256, 512])
def test_moe_config_128_experts_top8_768x2048(T):
    E, N, K, top_k = 128, 768, 2048, 8
    ids = syn.zipf_ids(syn.rng(1004 + T), T, E, top_k, 1.1)
    tok = np.arange(0, T, max(1, T // 8))
    got, ref = _run(syn.Q4_K, E, N, K, T, top_k, ids, seed=1004, token_rows=tok)
    U.check_close(got[tok].reshape(-1, N), ref[tok].reshape(-1, N), "bf16")


def test_moe_full_width_tiles_give_the_same_output(monkeypatch):
    # the comparison switch only widens the MMAs over columns no row fills
    E, N, K, T, top_k = 16, 256, 512, 40, 4
    ids = syn.zipf_ids(syn.rng(77), T, E, top_k, 1.1)
    got, ref = _run(syn.Q4_K, E, N, K, T, top_k, ids)
    monkeypatch.setenv("GGUF_MM_MOE_FULL_TILES", "1")
    got_full, _ = _run(syn.Q4_K, E, N, K, T, top_k, ids)
    U.check_close(got_full.reshape(-1, N), ref.reshape(-1, N), "bf16")
    assert np.array_equal(got_full, got)


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K, syn.Q4_0, syn.Q4_1, syn.Q5_0])
def test_moe_one_cta_per_sm_arm(qtype, monkeypatch):
    # the grouped GEMM of these formats runs two CTAs per SM (each with one MMA
    # issuer); the comparison arm keeps one per SM (two issuers) -- both against
    # the oracle, on tiles with a residual and ragged token columns
    E, N, K, T, top_k = 12, 384, 1024, 70, 4
    ids = syn.zipf_ids(syn.rng(78), T, E, top_k, 1.1)
    got, ref = _run(qtype, E, N, K, T, top_k, ids, residual=True)
    U.check_close(got.reshape(-1, N), ref.reshape(-1, N), "bf16")
    monkeypatch.setenv("GGUF_MM_MOE_CTAS", "1")
    got1, ref1 = _run(qtype, E, N, K, T, top_k, ids, residual=True)
    U.check_close(got1.reshape(-1, N), ref1.reshape(-1, N), "bf16")


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q8_0])
def test_moe_per_slot_activations(qtype):
    # down-projection form: every (token, slot) row has its own activations
    E, N, K, T, top_k = 8, 256, 512, 37, 4
    rs = syn.rng(91 + qtype)
    wE = syn.weight_blocks(rs, qtype, E * N, K)
    x = syn.normal(rs, (T, top_k, K), "bf16")
    r = syn.normal(rs, (T, top_k, N), "bf16")
    ids = _distinct_ids(syn.rng(92), T, E, top_k)
    y = torch.full((T, top_k, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_ID, qtype, N, K, T, E, top_k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    g.gguf_mm_id_slots(U.dev(wE), qtype, E, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, T, U.dev(ids), top_k,
                       U.dev(r, "bf16"), y, g.GGUF_DT_BF16, ws, ws_bytes)
    torch.cuda.synchronize()
    assert g.gguf_mm_check_errors() == 0
    if mv_form(qtype, T * top_k):
        ref = O.moe_mv_id_int8(wE, qtype, E, N, K, U.act_f32(x, "bf16"), ids, U.act_f64(r, "bf16"))
    else:
        ref = O.moe_mm_id_exact(wE, qtype, E, N, K, U.act_f64(x, "bf16"), ids, U.act_f64(r, "bf16"))
    U.check_close(U.host64(y).reshape(-1, N), ref.reshape(-1, N), "bf16")


def test_moe_per_slot_with_repeated_rows_equals_shared_rows():
    E, N, K, T, top_k = 8, 128, 256, 20, 3
    rs = syn.rng(93)
    wE = U.dev(syn.weight_blocks(rs, syn.Q5_K, E * N, K))
    x = syn.normal(rs, (T, K), "bf16")
    xs = np.repeat(x[:, None, :], top_k, axis=1)
    ids = U.dev(_distinct_ids(syn.rng(94), T, E, top_k))
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_ID, syn.Q5_K, N, K, T, E, top_k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    ys = []
    for fn, xin in ((g.gguf_mm_id, x), (g.gguf_mm_id_slots, xs)):
        y = torch.empty((T, top_k, N), dtype=torch.bfloat16, device="cuda")
        fn(wE, syn.Q5_K, E, N, K, U.dev(xin, "bf16"), g.GGUF_DT_BF16, T, ids, top_k, None, y, g.GGUF_DT_BF16, ws,
           ws_bytes)
        torch.cuda.synchronize()
        ys.append(U.host64(y))
    assert g.gguf_mm_check_errors() == 0
    assert np.array_equal(ys[0], ys[1])


@pytest.mark.parametrize("qtype", [syn.Q8_0, syn.Q6_K, syn.Q4_0, syn.Q4_1, syn.Q5_0, syn.Q5_1, syn.Q2_K, syn.Q3_K])
@pytest.mark.parametrize("T,top_k,per_slot", [(1, 8, False), (3, 4, True), ("limit", 8, False)])
def test_moe_decode_form_other_formats(qtype, T, top_k, per_slot):
    # the staged GEMV kernel in routed mode: every routed row an int8 GEMV of its
    # activation row against its expert; an invalid id leaves its row untouched.
    # "limit": the largest batch of this format that takes the decode form
    if T == "limit":
        T = U.moe_mv_max_rows(qtype) // top_k
    assert mv_form(qtype, T * top_k)
    E, N, K = 24, 320, 1024
    rs = syn.rng(310 + T * top_k + qtype)
    wE = syn.weight_blocks(rs, qtype, E * N, K)
    x = syn.normal(rs, (T, top_k, K) if per_slot else (T, K), "bf16")
    r = syn.normal(rs, (T, top_k, N), "f32")                 # the residual has y's type (f32)
    ids = syn.zipf_ids(syn.rng(311 + T), T, E, top_k, 1.1)
    ids[0, -1] = E + 3
    y = U.guarded((T, top_k, N), torch.float32, fill=float("nan"))
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_ID, qtype, N, K, T, E, top_k)
    ws = U.workspace(ws_bytes)
    fn = g.gguf_mm_id_slots if per_slot else g.gguf_mm_id
    fn(U.dev(wE), qtype, E, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, T, U.dev(ids), top_k, U.dev(r), y.t,
       g.GGUF_DT_F32, ws.t, ws_bytes)
    torch.cuda.synchronize()
    y.check("y")
    ws.check("workspace")
    assert g.gguf_mm_check_errors() == 0
    ref = O.moe_mv_id_int8(wE, qtype, E, N, K, U.act_f32(x, "bf16"), ids, r.astype(np.float64))
    U.check_close(U.host64(y.t).reshape(-1, N), ref.reshape(-1, N), "f32", allow_nan=True)


@pytest.mark.parametrize("T,top_k,per_slot", [(1, 8, False), (2, 8, True), (16, 8, False), (3, 5, True)])
@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K])
def test_moe_decode_form_128_experts_768x2048(qtype, T, top_k, per_slot):
    # decode: a few routed rows, each its own int8 GEMV (no routing)
    E, N, K = 128, 768, 2048
    rs = syn.rng(300 + T * top_k + qtype)
    wE = syn.weight_blocks(rs, qtype, E * N, K)
    x = syn.normal(rs, (T, top_k, K) if per_slot else (T, K), "bf16")
    r = syn.normal(rs, (T, top_k, N), "bf16")
    ids = syn.zipf_ids(syn.rng(301 + T), T, E, top_k, 1.1)
    assert mv_form(qtype, T * top_k)
    y = torch.full((T, top_k, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_ID, qtype, N, K, T, E, top_k)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    fn = g.gguf_mm_id_slots if per_slot else g.gguf_mm_id
    fn(U.dev(wE), qtype, E, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, T, U.dev(ids), top_k, U.dev(r, "bf16"), y,
       g.GGUF_DT_BF16, ws, ws_bytes)
    torch.cuda.synchronize()
    assert g.gguf_mm_check_errors() == 0
    ref = O.moe_mv_id_int8(wE, qtype, E, N, K, U.act_f32(x, "bf16"), ids, U.act_f64(r, "bf16"))
    U.check_close(U.host64(y).reshape(-1, N), ref.reshape(-1, N), "bf16")


@pytest.mark.parametrize("T,E,top_k", [(256, 128, 8), (5, 16, 3), (600, 4, 2)])
def test_moe_routing_tables_match_the_oracle(T, E, top_k):
    # the routing step's integer tables: per-expert offsets bit for bit against
    # the oracle's counts, the (expert, <= 128-row tile) work list in expert
    # order, and every expert's group holding exactly its routed entries
    ids = syn.zipf_ids(syn.rng(500 + T), T, E, top_k, 1.1)
    ids[0, 0], ids[T - 1, top_k - 1] = -3, E
    entries = T * top_k
    max_tiles = min(E, entries) + -(-entries // 128)
    offsets = U.guarded((E + 1,), torch.int32, fill=-7)
    ntiles = U.guarded((1,), torch.int32, fill=-7)
    tiles = U.guarded((max_tiles, 4), torch.int32, fill=-7)
    rows = U.guarded((entries,), torch.int32, fill=-7)
    g.gguf_mm_debug_moe_route(U.dev(ids.astype(np.int32)), entries, E, offsets.t, ntiles.t, tiles.t, max_tiles,
                              rows.t)
    torch.cuda.synchronize()
    for b, nm in ((offsets, "offsets"), (ntiles, "ntiles"), (tiles, "tiles"), (rows, "rows")):
        b.check(nm)
    counts, offs = O.moe_routing(ids, E)
    got_off = offsets.t.cpu().numpy().astype(np.int64)
    assert np.array_equal(got_off[:E], offs)
    assert got_off[E] == counts.sum()
    want_tiles = [(e, s0, min(128, int(counts[e]) - s0), 0) for e in range(E) for s0 in range(0, int(counts[e]), 128)]
    assert int(ntiles.t.item()) == len(want_tiles)
    assert [tuple(t) for t in tiles.t.cpu().numpy()[:len(want_tiles)].tolist()] == want_tiles
    got_rows = rows.t.cpu().numpy()
    flat = ids.ravel()
    for e in range(E):
        group = got_rows[offs[e]:offs[e] + counts[e]]
        assert sorted(group.tolist()) == np.flatnonzero(flat == e).tolist()


@pytest.mark.parametrize("T,top_k", [(70, 2), (9, 2)])
@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q8_0])
def test_moe_activation_rows_beyond_f16_range(qtype, T, top_k):
    # bf16 rows reaching 3e5, 1e20 and down to 1e-7 (f16 holds 6.1e-5 .. 65504):
    # each gathered row is scaled by a power of two into f16's range and the
    # epilogue scales its sums back; every row is checked against its own scale
    E, N, K = 8, 128, 512
    rs = syn.rng(55 + T + qtype)
    wE = syn.weight_blocks(rs, qtype, E * N, K)
    x32 = rs.standard_normal((T, K)).astype(np.float32)
    x32[0] *= 3e5
    x32[1] *= 1e20
    x32[2] *= 1e-7
    x32[3, ::7] *= 1e5
    x = syn.f32_to_bf16_bits(x32)
    ids = _distinct_ids(syn.rng(56), T, E, top_k)
    y = U.guarded((T, top_k, N), torch.float32)
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_ID, qtype, N, K, T, E, top_k)
    ws = U.workspace(ws_bytes)
    g.gguf_mm_id(U.dev(wE), qtype, E, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, T, U.dev(ids), top_k, None, y.t,
                 g.GGUF_DT_F32, ws.t, ws_bytes)
    torch.cuda.synchronize()
    y.check("y")
    assert g.gguf_mm_check_errors() == 0
    got = U.host64(y.t)
    if mv_form(qtype, T * top_k):
        ref = O.moe_mv_id_int8(wE, qtype, E, N, K, U.act_f32(x, "bf16"), ids)
        rel = 1e-4
    else:
        ref = O.moe_mm_id_exact(wE, qtype, E, N, K, U.act_f64(x, "bf16"), ids)
        rel = 2e-3
    for t in range(T):
        U.check_close(got[t], ref[t], "f32", rel=rel, what=f"token {t}")


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q5_K])
@pytest.mark.parametrize("T,top_k,per_slot", [(1, 8, 0), (3, 2, 0), (16, 8, 0), (4, 4, 1), (60, 2, 1)])
def test_moe_decode_form_integer_terms_bit_exact(qtype, T, top_k, per_slot):
    """The decode form's integer intermediates, row by routed row: the
    activation codes, scales and sums (in-kernel quantizer at <= 8 routed rows,
    the shared image above) and every sub-block dot against the row's expert
    equal the int8-path oracle's bit for bit (OpenVINO PR #39119
    "Implementation", GEMV row, applied per routed row as mul_mv_id does)."""
    E, N, K = 12, 96, 1024
    rs = syn.rng(900 + qtype + T + per_slot)
    wE = syn.weight_blocks(rs, qtype, E * N, K)
    ids = _distinct_ids(rs, T, E, top_k)
    ids[0, -1] = -1                                          # an invalid id: its row is left alone
    entries = T * top_k
    xrows = entries if per_slot else T
    x = syn.normal(rs, (xrows, K), "bf16")
    qa = torch.zeros((entries, K), dtype=torch.int8, device="cuda")
    da = torch.zeros((entries, K // 32), dtype=torch.float32, device="cuda")
    s = torch.zeros((entries, K // 32), dtype=torch.int32, device="cuda")
    D = U.guarded((entries, N, K // 32), torch.int32, fill=-999999)
    y = U.guarded((T, top_k, N), torch.float32)
    nws = g.gguf_mm_workspace_size(g.GGUF_OP_ID, qtype, N, K, T, E, top_k)
    ws = U.workspace(nws)
    g.gguf_mm_debug_moe_mv_terms(U.dev(wE), qtype, E, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, T, U.dev(ids), top_k,
                                 per_slot, None, y.t, g.GGUF_DT_F32, qa, da, s, D.t, ws.t, nws)
    torch.cuda.synchronize()
    for b, nm in ((D, "D"), (y, "y"), (ws, "workspace")):
        b.check(nm)
    assert g.gguf_mm_check_errors() == 0
    qa, da, s, Dh = qa.cpu().numpy(), da.cpu().numpy(), s.cpu().numpy(), D.t.cpu().numpy()
    x32 = U.act_f32(x, "bf16")
    rb = K // 256 * syn.BLOCK_BYTES[qtype]
    wv = wE.reshape(E, N, rb)
    for p, e in enumerate(ids.reshape(-1)):
        if e < 0:
            assert np.all(Dh[p] == -999999), "a row without an expert was written"
            continue
        arow = p if per_slot else p // top_k
        _, t = O.gemv_int8_path(wv[e], qtype, N, K, x32[arow:arow + 1], return_terms=True)
        assert np.array_equal(qa[p], t["qa"][0]), p
        assert np.array_equal(da[p], t["d_a"][0]), p
        assert np.array_equal(s[p], t["s"][0]), p
        assert np.array_equal(Dh[p].astype(np.int64), t["D"][0]), f"row {p}: D differs at {np.argwhere(Dh[p] != t['D'][0])[:5]}"


def test_moe_decode_form_terms_hook_refuses_the_routed_path():
    E, N, K, T, top_k = 4, 64, 256, 40, 4          # 160 routed rows: above the decode form
    ids = np.zeros((T, top_k), np.int32)
    nws = g.gguf_mm_workspace_size(g.GGUF_OP_ID, syn.Q4_K, N, K, T, E, top_k)
    ws = U.workspace(nws)
    w = U.dev(np.zeros(E * N * K // 256 * 144, np.uint8))
    x = torch.zeros((T, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((T, top_k, N), dtype=torch.float32, device="cuda")
    with pytest.raises(g.GGUFError) as e:
        g.gguf_mm_debug_moe_mv_terms(w, syn.Q4_K, E, N, K, x, g.GGUF_DT_BF16, T, U.dev(ids), top_k, 0, None, y,
                                     g.GGUF_DT_F32, workspace=ws.t, ws_bytes=nws)
    assert e.value.status == g.GGUF_ERR_UNSUPPORTED


def _run_path(qtype, E, N, K, T, top_k, wE, x, ids, path):
    y = U.guarded((T, top_k, N), torch.float32, fill=float("nan"))
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_ID, qtype, N, K, T, E, top_k)
    ws = U.workspace(ws_bytes, 0x6B)
    g.gguf_mm_id_path(U.dev(wE), qtype, E, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, T, U.dev(ids), top_k, 0, None,
                      y.t, g.GGUF_DT_F32, ws.t, ws_bytes, path)
    torch.cuda.synchronize()
    y.check("y")
    ws.check("workspace")
    assert g.gguf_mm_check_errors() == 0
    return U.host64(y.t)


@pytest.mark.parametrize("qtype", [syn.Q4_K, syn.Q8_0])
def test_moe_form_chosen_by_the_caller(qtype):
    # gguf_mm_id_path: AUTO is gguf_mm_id bit for bit; GEMV forces the decode form
    # (int8 path) and FUSED the routed tensor-core path, each where the batch-size
    # rule would take the other; GEMV above 128 routed rows is refused
    E, N, K, top_k = 8, 256, 512, 4
    rs = syn.rng(520 + qtype)
    wE = syn.weight_blocks(rs, qtype, E * N, K)
    for T in (2, 10):                                        # 8 and 40 routed rows
        x = syn.normal(rs, (T, K), "bf16")
        ids = _distinct_ids(rs, T, E, top_k)
        auto = _run_path(qtype, E, N, K, T, top_k, wE, x, ids, g.GGUF_PATH_AUTO)
        y = U.guarded((T, top_k, N), torch.float32, fill=float("nan"))
        ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_ID, qtype, N, K, T, E, top_k)
        ws = U.workspace(ws_bytes, 0x6B)
        g.gguf_mm_id(U.dev(wE), qtype, E, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, T, U.dev(ids), top_k, None, y.t,
                     g.GGUF_DT_F32, ws.t, ws_bytes)
        torch.cuda.synchronize()
        assert np.array_equal(auto, U.host64(y.t))
        dec = _run_path(qtype, E, N, K, T, top_k, wE, x, ids, g.GGUF_PATH_GEMV)
        U.check_close(dec.reshape(-1, N), O.moe_mv_id_int8(wE, qtype, E, N, K, U.act_f32(x, "bf16"), ids).reshape(-1, N),
                      "f32", what=f"decode form T={T}")
        rt = _run_path(qtype, E, N, K, T, top_k, wE, x, ids, g.GGUF_PATH_FUSED)
        U.check_close(rt.reshape(-1, N), O.moe_mm_id_exact(wE, qtype, E, N, K, U.act_f64(x, "bf16"), ids).reshape(-1, N),
                      "f32", rel=2e-3, what=f"routed T={T}")
        assert np.array_equal(auto, dec if mv_form(qtype, T * top_k) else rt)
    T = 40                                                   # 160 routed rows
    x = syn.normal(rs, (T, K), "bf16")
    ids = _distinct_ids(rs, T, E, top_k)
    ws_bytes = g.gguf_mm_workspace_size(g.GGUF_OP_ID, qtype, N, K, T, E, top_k)
    ws = U.workspace(ws_bytes)
    y = torch.empty((T, top_k, N), dtype=torch.float32, device="cuda")
    with pytest.raises(g.GGUFError) as err:
        g.gguf_mm_id_path(U.dev(wE), qtype, E, N, K, U.dev(x, "bf16"), g.GGUF_DT_BF16, T, U.dev(ids), top_k, 0,
                          None, y, g.GGUF_DT_F32, ws.t, ws_bytes, g.GGUF_PATH_GEMV)
    assert err.value.status == g.GGUF_ERR_UNSUPPORTED
    assert g.gguf_mm_check_errors() == 0
