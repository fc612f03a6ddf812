"""Pins for the CPU oracle: hand-worked blocks, bit-pattern invariants, exact
rational brute force, and special cases where the int8 path reduces to the plain
matmul.  CPU only."""
from fractions import Fraction

import numpy as np
import pytest

import gguf_synth as syn
from oracle import gguf_oracle as O
from tests import golden_blocks as gb


# ---------------------------------------------------------------- hand-worked blocks

@pytest.mark.parametrize("builder,decoder", [
    (gb.q4_k, O.dequant_q4_k), (gb.q5_k, O.dequant_q5_k), (gb.q6_k, O.dequant_q6_k), (gb.q2_k, O.dequant_q2_k),
    (gb.q3_k, O.dequant_q3_k)])
def test_hand_worked_kquant_blocks(builder, decoder):
    blk, expected = builder()
    w = decoder(blk[None, :])[0]
    for e, v in expected.items():
        assert w[e] == v, (e, w[e], v)


@pytest.mark.parametrize("builder,decoder", [
    (gb.q4_0, O.dequant_q4_0), (gb.q4_1, O.dequant_q4_1), (gb.q5_0, O.dequant_q5_0), (gb.q5_1, O.dequant_q5_1)])
def test_hand_worked_32_value_blocks(builder, decoder):
    blk, expected = builder()
    w = decoder(blk[None, :])[0]
    for e, v in expected.items():
        assert w[e] == v, (e, w[e], v)


def test_hand_worked_q8_0_blocks():
    for blk, expected in gb.q8_0():
        w = O.dequant_q8_0(blk[None, :])[0]
        for e, v in expected.items():
            assert w[e] == v, (e, w[e], v)


def test_decode_6bit_fields_all_distinct_bits():
    # each of the 16 six-bit fields set alone to 63 must light exactly one field
    for i in range(16):
        s = np.zeros((1, 12), np.uint8)
        j, is_min = i % 8, i >= 8
        if j < 4:
            s[0, j + 4 * is_min] = 63
        else:
            s[0, j + 4] = 0xF0 if is_min else 0x0F
            s[0, j - 4 + 4 * is_min] = 0xC0
        vals = [int(O.decode_6bit(s, k)[0]) for k in range(16)]
        assert vals[i] == 63 and sum(vals) == 63, (i, vals)


# ---------------------------------------------------------------- invariants

def _blocks_of(qtype, fill):
    return np.full((3, syn.BLOCK_BYTES[qtype]), fill, np.uint8)


def _set_f16(blk, off, val):
    blk[:, off:off + 2] = np.array([val], np.float16).view(np.uint8)


@pytest.mark.parametrize("qtype", [O.Q4_0, O.Q4_1, O.Q5_0, O.Q5_1, O.Q8_0, O.Q2_K, O.Q3_K, O.Q4_K, O.Q5_K, O.Q6_K])
def test_all_zero_blocks_decode_to_zero(qtype):
    w = O._DECODERS[qtype](_blocks_of(qtype, 0))
    assert np.all(w == 0)


@pytest.mark.parametrize("qtype,value", [(O.Q4_K, 882.0), (O.Q5_K, 1890.0), (O.Q6_K, -31.0),
                                         (O.Q8_0, -1.0), (O.Q4_0, 7.0), (O.Q4_1, 16.0), (O.Q5_0, 15.0),
                                         (O.Q5_1, 32.0), (O.Q2_K, 30.0), (O.Q3_K, 93.0)])
def test_all_max_bit_patterns(qtype, value):
    # all quant/scale bytes 0xFF, d = dmin = 1: sc = m = 63 and q at its maximum;
    # 32-value formats: q = 15 (31 with the fifth bit), d = m = 1:
    # (15 - 8), 15 + 1, (31 - 16), 31 + 1; Q2_K: sc = m = 15, q = 3: 15*3 - 15;
    # Q3_K: scale6 = 63, every hmask bit set, q = 3: (63 - 32) * 3
    blk = _blocks_of(qtype, 0xFF)
    if qtype == O.Q2_K:
        _set_f16(blk, 80, 1.0)
        _set_f16(blk, 82, 1.0)
    elif qtype == O.Q3_K:
        _set_f16(blk, 108, 1.0)
    elif qtype in (O.Q8_0, O.Q4_0, O.Q5_0):
        _set_f16(blk, 0, 1.0)
    elif qtype in (O.Q4_1, O.Q5_1):
        _set_f16(blk, 0, 1.0)
        _set_f16(blk, 2, 1.0)
    elif qtype == O.Q6_K:
        _set_f16(blk, 208, 1.0)
    else:
        _set_f16(blk, 0, 1.0)
        _set_f16(blk, 2, 1.0)
    w = O._DECODERS[qtype](blk)
    assert np.all(w == value)


def test_q6k_zero_quants_give_minus_32_d_sc():
    g = syn.rng(5)
    blk = syn.weight_blocks(g, O.Q6_K, 4, 256).reshape(4, 210)
    blk[:, 0:192] = 0
    w = O.dequant_q6_k(blk)
    d = O.f16_field(blk[:, 208:210])
    sc = blk[:, 192:208].view(np.int8).astype(np.float64)
    for e in range(256):
        assert np.array_equal(w[:, e], -32 * d * sc[:, e // 16])


@pytest.mark.parametrize("qtype", [O.Q4_0, O.Q4_1, O.Q5_0, O.Q5_1, O.Q8_0, O.Q2_K, O.Q3_K, O.Q4_K, O.Q5_K, O.Q6_K])
def test_scaling_d_by_power_of_two_scales_w(qtype):
    g = syn.rng(7)
    w = syn.weight_blocks(g, qtype, 2, 256)
    blk = w.reshape(-1, syn.BLOCK_BYTES[qtype]).copy()
    base = O._DECODERS[qtype](blk)
    offs = {O.Q8_0: [0], O.Q4_K: [0, 2], O.Q5_K: [0, 2], O.Q6_K: [208], O.Q4_0: [0], O.Q5_0: [0],
            O.Q4_1: [0, 2], O.Q5_1: [0, 2], O.Q2_K: [80, 82], O.Q3_K: [108]}[qtype]
    for off in offs:
        d = blk[:, off:off + 2].copy().view(np.float16)[:, 0]
        blk[:, off:off + 2] = (d * np.float16(4)).astype(np.float16).view(np.uint8).reshape(-1, 2)
    assert np.array_equal(O._DECODERS[qtype](blk), 4 * base)


def test_synthetic_blocks_follow_the_recipe():
    g = syn.rng(11)
    w6 = syn.weight_blocks(g, O.Q6_K, 16, 1024).reshape(-1, 210)
    sc = w6[:, 192:208].view(np.int8)
    assert sc.min() >= -32 and sc.max() <= 31
    w8 = syn.weight_blocks(g, O.Q8_0, 16, 1024).reshape(-1, 34)
    q = w8[:, 2:].view(np.int8)
    assert q.min() >= -127 and q.max() <= 127
    d = O.f16_field(w8[:, 0:2])
    assert np.all(d >= 0) and np.all(np.isfinite(d))


# ---------------------------------------------------------------- matmul vs exact rationals

@pytest.mark.parametrize("qtype", [O.Q4_0, O.Q4_1, O.Q5_0, O.Q5_1, O.Q8_0, O.Q2_K, O.Q3_K, O.Q4_K, O.Q5_K, O.Q6_K])
def test_matmul_exact_vs_fraction_brute_force(qtype):
    g = syn.rng(100 + qtype)
    N, K, M = 3, 256, 2
    w = syn.weight_blocks(g, qtype, N, K)
    x = syn.normal(g, (M, K), "f32").astype(np.float64)
    r = syn.normal(g, (M, N), "f32").astype(np.float64)
    w64 = O.dequant(w, qtype, N, K)
    ref = O.matmul_exact(x, w64, r)
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += Fraction(float(x[m, k])) * Fraction(float(w64[n, k]))
            acc += Fraction(float(r[m, n]))
            assert abs(ref[m, n] - float(acc)) <= 1e-12 * max(1.0, abs(float(acc)))


def test_dequant_row_major_block_order():
    # a row of 2 blocks: decoding row-wise must equal decoding each block alone
    g = syn.rng(3)
    w = syn.weight_blocks(g, O.Q4_K, 2, 512)
    w64 = O.dequant(w, O.Q4_K, 2, 512)
    for n in range(2):
        for kb in range(2):
            blk = w[n, kb * 144:(kb + 1) * 144][None, :]
            assert np.array_equal(w64[n, kb * 256:(kb + 1) * 256], O.dequant_q4_k(blk)[0])


# ---------------------------------------------------------------- activation quantizer

def test_act_quant_constant_blocks_hit_127():
    x = np.zeros((2, 64), np.float32)
    x[0, :32] = 0.3
    x[0, 32:] = -7.25
    x[1, :32] = 1e-20
    qa, d_a, s = O.quantize_act_q8(x)
    assert np.all(qa[0, :32] == 127) and np.all(qa[0, 32:] == -127)
    assert np.all(qa[1, :32] == 127)
    assert d_a[0, 0] == np.float32(0.3) / np.float32(127)
    assert s[0, 0] == 127 * 32 and s[0, 1] == -127 * 32


def test_act_quant_zero_block():
    qa, d_a, s = O.quantize_act_q8(np.zeros((1, 32), np.float32))
    assert np.all(qa == 0) and d_a[0, 0] == 0 and s[0, 0] == 0


def test_act_quant_exact_multiples_roundtrip():
    g = syn.rng(21)
    n = g.integers(-127, 128, size=(3, 96))
    n[:, ::32] = 127                                   # amax = 127 * 2**-3 in every block
    x = (n * 2.0 ** -3).astype(np.float32)
    qa, d_a, s = O.quantize_act_q8(x)
    assert np.all(d_a == np.float32(2.0 ** -3))
    assert np.array_equal(qa.astype(np.int64), n)
    assert np.array_equal(s, n.reshape(3, 3, 32).sum(axis=2))


def test_act_quant_rounds_half_away_from_zero():
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 127.0                                    # d_a = 1, id = 1
    x[0, 1], x[0, 2], x[0, 3], x[0, 4] = 2.5, -2.5, 0.5, -0.5
    qa, d_a, _ = O.quantize_act_q8(x)
    assert d_a[0, 0] == 1.0
    assert list(qa[0, 1:5]) == [3, -3, 1, -1]


# ---------------------------------------------------------------- int8 path reduces to the plain matmul

@pytest.mark.parametrize("qtype", [O.Q4_0, O.Q4_1, O.Q5_0, O.Q5_1, O.Q8_0, O.Q2_K, O.Q3_K, O.Q4_K, O.Q5_K, O.Q6_K])
def test_int8_path_equals_exact_when_activations_are_on_the_grid(qtype):
    # x = d_a * integers with amax = 127 * d_a in every block: quantization is
    # lossless, so the int8-path result must equal the exact matmul
    g = syn.rng(40 + qtype)
    N, K, M = 5, 512, 3
    w = syn.weight_blocks(g, qtype, N, K)
    n = g.integers(-127, 128, size=(M, K))
    n[:, ::32] = -127
    scale = 2.0 ** g.integers(-6, 2, size=(M, K // 32, 1))
    x = (n.reshape(M, K // 32, 32) * scale).reshape(M, K).astype(np.float32)
    r = syn.normal(g, (M, N), "f32")
    y8 = O.gemv_int8_path(w, qtype, N, K, x, r)
    ref = O.matmul_exact(x, O.dequant(w, qtype, N, K), r)
    assert np.max(np.abs(y8 - ref)) <= 1e-12 * np.max(np.abs(ref))


@pytest.mark.parametrize("qtype", [O.Q4_0, O.Q4_1, O.Q5_0, O.Q5_1, O.Q8_0, O.Q2_K, O.Q3_K, O.Q4_K, O.Q5_K, O.Q6_K])
def test_int8_path_close_to_exact_on_normal_data(qtype):
    # the activation rounding error is the only gap: RMS ~ amax/(127*sqrt(12)) per value
    g = syn.rng(60 + qtype)
    N, K, M = 16, 1024, 2
    w = syn.weight_blocks(g, qtype, N, K)
    x = syn.normal(g, (M, K), "f32")
    y8 = O.gemv_int8_path(w, qtype, N, K, x)
    ref = O.matmul_exact(x, O.dequant(w, qtype, N, K))
    assert np.max(np.abs(y8 - ref)) <= 3e-2 * np.max(np.abs(ref))
    assert np.max(np.abs(y8 - ref)) > 0


@pytest.mark.parametrize("qtype", [O.Q4_0, O.Q4_1, O.Q5_0, O.Q5_1, O.Q8_0, O.Q2_K, O.Q3_K, O.Q4_K, O.Q5_K, O.Q6_K])
def test_integer_terms_rebuild_the_decoded_weights(qtype):
    g = syn.rng(80 + qtype)
    N, K = 3, 512
    w = syn.weight_blocks(g, qtype, N, K)
    q_w, sub, scale, minv = O.weight_int_terms(w, qtype, N, K)
    rebuilt = np.repeat(scale, sub, axis=1) * q_w - np.repeat(minv, sub, axis=1)
    assert np.array_equal(rebuilt, O.dequant(w, qtype, N, K))


def test_int8_dots_brute_force_tiny():
    g = syn.rng(90)
    q_w = g.integers(-32, 32, size=(2, 64))
    qa = g.integers(-127, 128, size=(3, 64)).astype(np.int8)
    D = O.int8_dots(q_w, 16, qa)
    for m in range(3):
        for n in range(2):
            for j in range(4):
                assert D[m, n, j] == sum(int(q_w[n, k]) * int(qa[m, k]) for k in range(16 * j, 16 * j + 16))


# ---------------------------------------------------------------- Q6_K planes

def test_q6k_planes_roundtrip_and_offsets():
    g = syn.rng(13)
    N, K = 6, 768
    w = syn.weight_blocks(g, O.Q6_K, N, K)
    nblk = N * K // 256
    p = O.q6k_to_planes(w)
    assert p.size == w.size == 210 * nblk                     # same size
    assert O.q6k_planes_offsets(nblk) == (0, 128 * nblk, 192 * nblk, 208 * nblk, 210 * nblk)
    back = O.q6k_from_planes(p, nblk)
    assert np.array_equal(back.reshape(N, -1), w)             # same contents
    blk = w.reshape(nblk, 210)
    for b in (0, 1, nblk - 1):                                 # field by field
        assert np.array_equal(p[128 * b:128 * b + 128], blk[b, 0:128])
        assert np.array_equal(p[128 * nblk + 64 * b:128 * nblk + 64 * b + 64], blk[b, 128:192])
        assert np.array_equal(p[192 * nblk + 16 * b:192 * nblk + 16 * b + 16], blk[b, 192:208])
        assert np.array_equal(p[208 * nblk + 2 * b:208 * nblk + 2 * b + 2], blk[b, 208:210])
    assert np.array_equal(O.dequant_q6k_planes(p, N, K), O.dequant(w, O.Q6_K, N, K))


# ---------------------------------------------------------------- decode-once padded buffer

def test_rounding_helpers_ties_to_even():
    one = 1.0
    assert O.round_f64_to_bf16_bits(np.array([one + 2 ** -8]))[0] == 0x3F80
    assert O.round_f64_to_bf16_bits(np.array([one + 3 * 2 ** -8]))[0] == 0x3F82
    assert O.round_f64_to_bf16_bits(np.array([one + 2 ** -8 + 2 ** -30]))[0] == 0x3F81
    assert O.round_f64_to_bf16_bits(np.array([-2.0, 0.0]))[0] == 0xC000
    assert O.round_f64_to_f16_bits(np.array([one + 2 ** -11]))[0] == 0x3C00
    assert O.round_f64_to_f16_bits(np.array([one + 3 * 2 ** -11]))[0] == 0x3C02
    # the sign of zero survives rounding
    assert list(O.round_f64_to_bf16_bits(np.array([-0.0, 0.0]))) == [0x8000, 0x0000]
    assert list(O.round_f64_to_f16_bits(np.array([-0.0, 0.0]))) == [0x8000, 0x0000]


def _nearest_bits_brute_force(v: float, all_vals: np.ndarray, all_bits: np.ndarray) -> int:
    """Nearest representable value by exhaustive search (exact rationals), ties
    to the even bit pattern."""
    from fractions import Fraction
    fv = Fraction(v)
    i = int(np.searchsorted(all_vals, v))
    best = None
    for j in (i - 1, i, i + 1):
        if 0 <= j < len(all_vals):
            d = abs(Fraction(float(all_vals[j])) - fv)
            key = (d, int(all_bits[j]) & 1)
            if best is None or key < best[0]:
                best = (key, int(all_bits[j]))
    return best[1]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_rounding_helpers_against_exhaustive_search(dtype):
    # every finite positive value of the type, sorted; random f64 inputs of
    # both signs within the normal and subnormal ranges
    bits = np.arange(0x0000, 0x7C00 if dtype == "f16" else 0x7F80, dtype=np.uint16)
    vals = bits.view(np.float16).astype(np.float64) if dtype == "f16" else O.bf16_bits_to_f64(bits)
    rs = np.random.default_rng(8)
    mag = rs.uniform(0.5, 2.0, 3000) * 2.0 ** rs.integers(-30 if dtype == "f16" else -140, 15, 3000)
    rnd = O.round_f64_to_f16_bits if dtype == "f16" else O.round_f64_to_bf16_bits
    got = rnd(mag)
    for v, gb in zip(mag, got):
        assert int(gb) == _nearest_bits_brute_force(float(v), vals, bits), (v, hex(int(gb)))
    assert np.array_equal(rnd(-mag), got | 0x8000)


@pytest.mark.parametrize("odt", ["f16", "bf16"])
def test_padding_changes_only_the_stride(odt):
    g = syn.rng(17)
    N, K = 4, 512
    w = syn.weight_blocks(g, O.Q8_0, N, K)
    packed = O.dequant_padded_bits(w, O.Q8_0, N, K, K, odt)
    padded = O.dequant_padded_bits(w, O.Q8_0, N, K, K + 64, odt)
    assert np.array_equal(padded[:, :K], packed)
    assert np.all(padded[:, K:] == 0)


# ---------------------------------------------------------------- MoE

def test_moe_with_one_expert_equals_dense():
    g = syn.rng(19)
    E, N, K, T, top_k = 3, 8, 256, 4, 2
    wE = syn.weight_blocks(g, O.Q4_K, E * N, K)
    x = syn.normal(g, (T, K), "f32")
    ids = np.zeros((T, top_k), np.int32)
    ids[:, 0], ids[:, 1] = 2, 1
    y = O.moe_mm_id_exact(wE, O.Q4_K, E, N, K, x, ids)
    rb = wE.shape[1]
    for slot, e in ((0, 2), (1, 1)):
        dense = O.matmul_exact(x, O.dequant(wE[e * N:(e + 1) * N].reshape(N, rb), O.Q4_K, N, K))
        assert np.max(np.abs(y[:, slot] - dense)) <= 1e-12 * np.max(np.abs(dense))


def test_moe_routing_counts_by_brute_force():
    # counts and offsets restated as explicit loops over every (token, slot),
    # including ids outside [0, n_expert), which select nothing
    g = syn.rng(23)
    E = 128
    ids = syn.zipf_ids(g, 64, E, 8)
    assert all(len(set(r)) == 8 for r in ids.tolist())
    ids[3, 2], ids[9, 0], ids[40, 7] = -1, E, E + 5
    counts, offsets = O.moe_routing(ids, E)
    for e in range(E):
        n = 0
        for t in range(ids.shape[0]):
            for k in range(ids.shape[1]):
                n += int(ids[t, k] == e)
        assert counts[e] == n
        before = 0
        for e2 in range(e):
            for t in range(ids.shape[0]):
                for k in range(ids.shape[1]):
                    before += int(ids[t, k] == e2)
        assert offsets[e] == before
    assert counts.sum() == 64 * 8 - 3
    assert counts[0] >= counts[64]                     # Zipf: low ranks hit more often


def test_moe_out_of_range_ids_select_no_expert():
    g = syn.rng(29)
    E, N, K = 2, 4, 256
    wE = syn.weight_blocks(g, O.Q8_0, E * N, K)
    x = syn.normal(g, (3, K), "f32")
    ids = np.array([[0], [-1], [E]], np.int32)
    y = O.moe_mm_id_exact(wE, O.Q8_0, E, N, K, x, ids)
    assert np.all(np.isfinite(y[0])) and np.all(np.isnan(y[1])) and np.all(np.isnan(y[2]))


def test_moe_per_slot_rows_reduce_to_shared_rows_and_to_dense():
    # per-slot activations that repeat the token's row give the shared-row
    # result; each slot's own row multiplies its own expert
    g = syn.rng(31)
    E, N, K, T, top_k = 3, 8, 256, 4, 2
    wE = syn.weight_blocks(g, O.Q4_K, E * N, K)
    x = syn.normal(g, (T, K), "f32")
    ids = np.array([[0, 2], [1, 0], [2, 1], [0, 1]], np.int32)
    shared = O.moe_mm_id_exact(wE, O.Q4_K, E, N, K, x, ids)
    assert np.array_equal(O.moe_mm_id_exact(wE, O.Q4_K, E, N, K, np.repeat(x[:, None, :], top_k, 1), ids), shared)
    xs = syn.normal(g, (T, top_k, K), "f32")
    y = O.moe_mm_id_exact(wE, O.Q4_K, E, N, K, xs, ids)
    rb = wE.shape[1]
    for t in range(T):
        for k in range(top_k):
            e = ids[t, k]
            dense = O.matmul_exact(xs[t, k][None, :], O.dequant(wE[e * N:(e + 1) * N].reshape(N, rb), O.Q4_K, N, K))
            assert np.max(np.abs(y[t, k] - dense[0])) <= 1e-12 * np.max(np.abs(dense))


def test_moe_decode_form_reduces_to_the_int8_gemv():
    # all slots on one expert with the token's shared row: every slot is that
    # expert's int8-path GEMV of the row; a per-slot row changes only its slot
    g = syn.rng(37)
    E, N, K, T, top_k = 3, 8, 256, 2, 2
    wE = syn.weight_blocks(g, O.Q5_K, E * N, K)
    x = syn.normal(g, (T, K), "f32")
    ids = np.full((T, top_k), 1, np.int32)
    y = O.moe_mv_id_int8(wE, O.Q5_K, E, N, K, x, ids)
    w1 = wE[N:2 * N]
    ref = O.gemv_int8_path(w1, O.Q5_K, N, K, x)
    for k in range(top_k):
        assert np.array_equal(y[:, k], ref)
    xs = np.repeat(x[:, None, :], top_k, 1)
    xs[1, 1] = syn.normal(g, (K,), "f32")
    ys = O.moe_mv_id_int8(wE, O.Q5_K, E, N, K, xs, ids)
    assert np.array_equal(ys[0], y[0]) and np.array_equal(ys[1, 0], y[1, 0])
    assert np.array_equal(ys[1, 1], O.gemv_int8_path(w1, O.Q5_K, N, K, xs[1, 1][None, :])[0])
    ids[0, 1] = -1
    assert np.all(np.isnan(O.moe_mv_id_int8(wE, O.Q5_K, E, N, K, x, ids)[0, 1]))


@pytest.mark.parametrize("qtype", [O.Q4_0, O.Q4_1, O.Q5_0, O.Q5_1])
def test_32_value_codes_by_bit_addressing(qtype):
    # element e's 4-bit code is bits 4*(e // 16) .. +3 of byte (e % 16) of the
    # code field, its fifth bit is bit e of the little-endian 32-bit qh word:
    # rebuilt here from unpacked bit arrays, compared with the decoders
    g = syn.rng(123 + qtype)
    blk = syn.weight_blocks(g, qtype, 4, 64).reshape(-1, syn.BLOCK_BYTES[qtype])
    q_off = {O.Q4_0: 2, O.Q4_1: 4, O.Q5_0: 6, O.Q5_1: 8}[qtype]
    bits = np.unpackbits(blk[:, q_off:q_off + 16], axis=1, bitorder="little").reshape(-1, 16, 8)
    hbits = np.unpackbits(blk[:, q_off - 4:q_off], axis=1, bitorder="little") if qtype in (O.Q5_0, O.Q5_1) else None
    d = O.f16_field(blk[:, 0:2])
    m = O.f16_field(blk[:, 2:4]) if qtype in (O.Q4_1, O.Q5_1) else 0.0
    w = O._DECODERS[qtype](blk)
    for e in range(32):
        lo = 4 * (e // 16)
        q = np.zeros(blk.shape[0], np.int64)
        for i in range(4):
            q = q + (bits[:, e % 16, lo + i].astype(np.int64) << i)
        if hbits is not None:
            q = q + 16 * hbits[:, e].astype(np.int64)
        want = {O.Q4_0: (q - 8) * d, O.Q5_0: (q - 16) * d}.get(qtype, q * d + m)
        assert np.array_equal(w[:, e], want), e


def test_q3k_zero_codes_give_minus_4_d_scale():
    # every 2-bit code and hmask bit 0: q3 = -4 everywhere, w = -4 * d * (scale6 - 32)
    g = syn.rng(9)
    blk = syn.weight_blocks(g, O.Q3_K, 4, 256).reshape(4, 110)
    blk[:, 0:96] = 0
    w = O.dequant_q3_k(blk)
    d = O.f16_field(blk[:, 108:110])
    for e in range(256):
        assert np.array_equal(w[:, e], -4 * d * (O.q3k_scale6(blk[:, 96:108], e // 16) - 32))


@pytest.mark.parametrize("qtype", [O.Q2_K, O.Q3_K])
def test_2_bit_codes_and_q3k_scales_by_bit_addressing(qtype):
    # element e = 128h + 32j + 16p + l: its code is bits 2j..2j+1 of qs byte
    # 32h + 16p + l, its Q3_K high bit is bit e // 32 of hmask byte e % 32, and
    # Q3_K scale i is assembled from unpacked bits of the 12 scale bytes: rebuilt
    # here from bit arrays and compared with the decoders
    g = syn.rng(321 + qtype)
    bb = syn.BLOCK_BYTES[qtype]
    blk = syn.weight_blocks(g, qtype, 4, 256).reshape(-1, bb)
    q_off = 16 if qtype == O.Q2_K else 32
    qbits = np.unpackbits(blk[:, q_off:q_off + 64], axis=1, bitorder="little").reshape(-1, 64, 8)
    w = O._DECODERS[qtype](blk)
    if qtype == O.Q2_K:
        d, dmin = O.f16_field(blk[:, 80:82]), O.f16_field(blk[:, 82:84])
        sc = blk[:, 0:16].astype(np.int64)
    else:
        d = O.f16_field(blk[:, 108:110])
        hbits = np.unpackbits(blk[:, 0:32], axis=1, bitorder="little").reshape(-1, 32, 8)
        sbits = np.unpackbits(blk[:, 96:108], axis=1, bitorder="little").reshape(-1, 12, 8)
    for e in range(256):
        h, r = divmod(e, 128)
        j, r2 = divmod(r, 32)
        byte = 32 * h + r2
        q = qbits[:, byte, 2 * j].astype(np.int64) + 2 * qbits[:, byte, 2 * j + 1].astype(np.int64)
        i = e // 16
        if qtype == O.Q2_K:
            want = d * (sc[:, i] & 15) * q - dmin * (sc[:, i] >> 4)
        else:
            q = q - 4 * (1 - hbits[:, e % 32, e // 32].astype(np.int64))
            lo_bits = range(0, 4) if i < 8 else range(4, 8)
            s6 = sum(sbits[:, i % 8, b].astype(np.int64) << k for k, b in enumerate(lo_bits))
            s6 = s6 + (sbits[:, 8 + i % 4, 2 * (i // 4)].astype(np.int64) << 4)
            s6 = s6 + (sbits[:, 8 + i % 4, 2 * (i // 4) + 1].astype(np.int64) << 5)
            want = d * (s6 - 32) * q
        assert np.array_equal(w[:, e], want), e
