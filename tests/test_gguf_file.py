"""The GGUF container reader (gguf_file_* in the C ABI): a hand-assembled file,
round trips through an independent writer, and malformed files.

GGUF Support Proposal for mobius, 1.1 "Overview" (one file: metadata
key-value pairs and tensors with a per-tensor type) and 1.3 (tensor names).
The byte layout is the published GGUF container layout, version 3; the
hand-typed fixture tests/golden/gguf_minimal.hex pins both the reader and the
writer the other tests use.  The reader is host code, so everything here but
the last test runs without a GPU."""
import os
import struct

import numpy as np
import pytest

import gguf_quant_weight_gb300 as g
import gguf_synth as syn
from oracle import gguf_oracle as O
from tests import gguf_writer as W

HERE = os.path.dirname(os.path.abspath(__file__))
QTYPES = [syn.Q8_0, syn.Q4_K, syn.Q5_K, syn.Q6_K, syn.Q4_0, syn.Q4_1, syn.Q5_0, syn.Q5_1, syn.Q2_K, syn.Q3_K]


@pytest.fixture(scope="module", autouse=True)
def lib():
    from gguf_quant_weight_gb300 import _build
    _build.build()
    return g.load_library()


def _fixture_bytes():
    with open(os.path.join(HERE, "golden", "gguf_minimal.hex")) as f:
        return bytes(int(t, 16) for line in f for t in line.split("#")[0].split())


def _put(tmp_path, data, name="f.gguf"):
    p = tmp_path / name
    p.write_bytes(data)
    return str(p)


def _status(path):
    try:
        with g.GGUFFile(path):
            return g.GGUF_OK
    except g.GGUFError as e:
        return e.status


def test_hand_assembled_file(tmp_path):
    with g.GGUFFile(_put(tmp_path, _fixture_bytes())) as f:
        assert f.version == 3 and f.alignment == 32
        assert f.keys() == [("general.architecture", W.STRING), ("llama.block_count", W.U32)]
        assert f.get_string("general.architecture") == "llama"
        assert f.get_int("llama.block_count") == 2
        assert f.get_float("llama.block_count") == 2.0
        assert f.tensors() == [("blk.0.attn_q.weight", 8, (32, 2))]
        assert f.tensor_info(0)[3:] == (192, 68)
        blocks, qt, N, K = f.weight("blk.0.attn_q.weight")
    assert (qt, N, K) == (syn.Q8_0, 2, 32) and blocks.shape == (2, 34)
    w = O.dequant(blocks, qt, N, K)
    assert np.array_equal(w[0], np.arange(32.0)) and np.all(w[1] == -0.5)


def test_writer_reproduces_the_hand_assembled_file():
    blocks = np.zeros((2, 34), np.uint8)
    blocks[0, :2] = [0x00, 0x3C]
    blocks[0, 2:] = np.arange(32)
    blocks[1, :2] = [0x00, 0x38]
    blocks[1, 2:] = 0xFF
    data = W.gguf_bytes([("general.architecture", W.STRING, "llama"), ("llama.block_count", W.U32, 2)],
                        [W.weight_tensor("blk.0.attn_q.weight", syn.Q8_0, blocks, 2, 32)])
    assert data == _fixture_bytes()


def _all_value_types():
    return [
        ("t.u8", W.U8, 250), ("t.i8", W.I8, -7), ("t.u16", W.U16, 65000), ("t.i16", W.I16, -30000),
        ("t.u32", W.U32, 4_000_000_000), ("t.i32", W.I32, -2_000_000_000), ("t.f32", W.F32, 0.15625),
        ("t.bool", W.BOOL, True), ("t.str", W.STRING, "grüße ∑"), ("t.u64", W.U64, 2**63 - 5),
        ("t.i64", W.I64, -2**62), ("t.f64", W.F64, -1e-300),
        ("t.arr_u32", W.ARRAY, (W.U32, [1, 2, 3, 2**32 - 1])), ("t.arr_f32", W.ARRAY, (W.F32, [0.5, -2.0])),
        ("t.arr_str", W.ARRAY, (W.STRING, ["<s>", "</s>", ""])), ("t.arr_empty", W.ARRAY, (W.I64, [])),
        ("t.empty_str", W.STRING, ""),
    ]


@pytest.mark.parametrize("alignment", [None, 64, 4096])
def test_round_trip_every_value_type_and_weight_format(tmp_path, alignment):
    rs = syn.rng(91)
    tensors, shapes = [], {}
    for i, qt in enumerate(QTYPES):
        N, K = 3 + i, (256 if syn.BLOCK_VALUES[qt] == 256 else 64) * (1 + i % 2)
        b = syn.weight_blocks(rs, qt, N, K)
        tensors.append(W.weight_tensor(f"blk.{i}.ffn_up.weight", qt, b, N, K))
        shapes[f"blk.{i}.ffn_up.weight"] = (b, qt, N, K)
    f32 = rs.standard_normal((5, 7)).astype(np.float32)
    f16 = rs.standard_normal((3, 2, 4)).astype(np.float16)
    tensors.append(("output_norm.weight", 0, (7, 5), f32.tobytes()))
    tensors.append(("t.f16", 1, (4, 2, 3), f16.tobytes()))
    kv = _all_value_types()
    path = str(tmp_path / "w.gguf")
    W.write(path, kv, tensors, alignment)
    with g.GGUFFile(path) as f:
        assert f.alignment == (alignment or 32)
        keys = dict(f.keys())
        for k, vt, v in kv:
            assert keys[k] == vt
            if vt in (W.F32, W.F64):
                assert f.get_float(k) == v
            elif vt == W.STRING:
                assert f.get_string(k) == v
            elif vt == W.ARRAY:
                et, items = v
                got = f.get_array(k)
                if et == W.STRING:
                    assert got == (W.STRING, len(items))
                else:
                    assert got.tolist() == items
            else:
                assert f.get_int(k) == int(v)
        for name, (b, qt, N, K) in shapes.items():
            got, qt2, N2, K2 = f.weight(name)
            assert (qt2, N2, K2) == (qt, N, K)
            assert np.array_equal(got, b)
            assert f.tensor_info(f.find_tensor(name))[3] % f.alignment == 0
        assert np.array_equal(f.tensor_bytes("output_norm.weight").view(np.float32).reshape(5, 7), f32)
        assert f.tensor_info(f.find_tensor("t.f16"))[2] == (4, 2, 3)
        assert np.array_equal(f.tensor_bytes("t.f16").view(np.float16).reshape(3, 2, 4), f16)
        with pytest.raises(g.GGUFError) as e:
            f.weight("output_norm.weight")              # f32: not a block-quantized weight
        assert e.value.status == g.GGUF_ERR_UNSUPPORTED


def test_lookups_and_type_mismatches(tmp_path):
    path = _put(tmp_path, W.gguf_bytes(_all_value_types(), []))
    with g.GGUFFile(path) as f:
        for call, key in ((f.get_int, "nope"), (f.get_string, "nope"), (f.find_tensor, "nope")):
            with pytest.raises(g.GGUFError) as e:
                call(key)
            assert e.value.status == g.GGUF_ERR_NOT_FOUND
        for call, key in ((f.get_int, "t.str"), (f.get_int, "t.f32"), (f.get_string, "t.u8"),
                          (f.get_array, "t.u8"), (f.get_int, "t.arr_u32")):
            with pytest.raises(g.GGUFError) as e:
                call(key)
            assert e.value.status == g.GGUF_ERR_UNSUPPORTED
        assert f.tensors() == []


def test_u64_above_int64_max_is_not_an_int(tmp_path):
    path = _put(tmp_path, W.gguf_bytes([("big", W.U64, 2**64 - 1)], []))
    with g.GGUFFile(path) as f:
        with pytest.raises(g.GGUFError) as e:
            f.get_int("big")
        assert e.value.status == g.GGUF_ERR_UNSUPPORTED


def test_every_truncation_is_a_format_error(tmp_path):
    data = _fixture_bytes()
    assert _status(_put(tmp_path, data)) == g.GGUF_OK
    for n in range(len(data)):
        assert _status(_put(tmp_path, data[:n])) == g.GGUF_ERR_FORMAT, n


def test_missing_file_is_an_io_error(tmp_path):
    assert _status(str(tmp_path / "absent.gguf")) == g.GGUF_ERR_IO
    assert _status(str(tmp_path)) in (g.GGUF_ERR_IO, g.GGUF_ERR_FORMAT)   # a directory


def _patched(data, at, fmt, value):
    b = bytearray(data)
    struct.pack_into(fmt, b, at, value)
    return bytes(b)


def test_malformed_headers(tmp_path):
    base = _fixture_bytes()
    bad = {
        "magic": _patched(base, 0, "<I", 0x46554746),
        "version 1": _patched(base, 4, "<I", 1),
        "version 4": _patched(base, 4, "<I", 4),
        "tensor count past the file": _patched(base, 8, "<Q", 2),
        "kv count past the file": _patched(base, 16, "<Q", 3),
        "huge kv count": _patched(base, 16, "<Q", 2**62),
        "key length past the file": _patched(base, 24, "<Q", 10**6),
        "huge key length": _patched(base, 24, "<Q", 2**64 - 1),
        "unknown value type": _patched(base, 52, "<I", 13),
        "string length past the file": _patched(base, 56, "<Q", 2**63),
        "n_dims 0": _patched(base, 129, "<I", 0),
        "n_dims 5": _patched(base, 129, "<I", 5),
        "dim 0": _patched(base, 133, "<Q", 0),
        "dims not a whole block": _patched(base, 133, "<Q", 48),
        "data past the file": _patched(base, 141, "<Q", 3),
        "offset not aligned": _patched(base, 153, "<Q", 8),
        "offset past the file": _patched(base, 153, "<Q", 2**63),
    }
    for what, data in bad.items():
        assert _status(_put(tmp_path, data)) == g.GGUF_ERR_FORMAT, what
    for a in (0, 3, 48, 1 << 21):
        data = W.gguf_bytes([], [], alignment=a) if a else W.gguf_bytes([("general.alignment", W.U32, 0)], [])
        assert _status(_put(tmp_path, data)) == g.GGUF_ERR_FORMAT, a
    assert _status(_put(tmp_path, W.gguf_bytes([("general.alignment", W.STRING, "32")], []))) == g.GGUF_ERR_FORMAT
    nested = W.gguf_bytes([("x", W.ARRAY, (W.U8, []))], [])
    nested = nested.replace(struct.pack("<IQ", W.U8, 0), struct.pack("<IQ", W.ARRAY, 1) + struct.pack("<IQ", W.U8, 0))
    assert _status(_put(tmp_path, nested)) == g.GGUF_ERR_FORMAT


def test_unknown_tensor_types_are_listed_but_not_read(tmp_path):
    data = W.gguf_bytes([], [("iq", 23, (256, 2), b"\0" * 64)])    # a type whose size the reader does not know
    with g.GGUFFile(_put(tmp_path, data)) as f:
        assert f.tensors() == [("iq", 23, (256, 2))]
        assert f.tensor_info(0)[4] == 0
        with pytest.raises(g.GGUFError) as e:
            f.tensor_bytes("iq")
        assert e.value.status == g.GGUF_ERR_UNSUPPORTED


def test_random_corruptions_never_read_out_of_bounds(tmp_path):
    """Seeded byte flips all over a file with every value type: each open gives
    OK or FORMAT, and an OK file answers every accessor."""
    rs = syn.rng(17)
    b = syn.weight_blocks(rs, syn.Q4_K, 2, 256)
    base = W.gguf_bytes(_all_value_types(), [W.weight_tensor("w", syn.Q4_K, b, 2, 256)])
    path = str(tmp_path / "c.gguf")
    n_ok = 0
    for it in range(1500):
        d = bytearray(base)
        for _ in range(1 + it % 4):
            d[int(rs.integers(0, len(d)))] = int(rs.integers(0, 256))
        if it % 5 == 0:
            d = d[:int(rs.integers(0, len(d)))]
        with open(path, "wb") as fh:
            fh.write(d)
        st = _status(path)
        assert st in (g.GGUF_OK, g.GGUF_ERR_FORMAT)
        if st == g.GGUF_OK:
            n_ok += 1
            with g.GGUFFile(path) as f:
                for k, vt in f.keys():
                    for call in (f.get_int, f.get_float, f.get_string, f.get_array):
                        try:
                            call(k)
                        except g.GGUFError:
                            pass
                for i, t in enumerate(f.tensors()):
                    if f.tensor_info(i)[4]:
                        f.tensor_bytes(i)
    assert n_ok > 0


@pytest.mark.gpu
@pytest.mark.parametrize("qtype", QTYPES)
def test_weights_read_from_a_file_run_on_the_gpu(tmp_path, qtype):
    """A weight read from a .gguf file goes to the matmul entry points as it is."""
    import torch
    from tests import gpu_util as U
    U.require_gpu()
    N, K, M = 384, 2048, 3   # raw Q6_K rows on the tensor-core path need K % 2048 == 0 (16-byte row pitch)
    rs = syn.rng(300 + qtype)
    b = syn.weight_blocks(rs, qtype, N, K)
    path = str(tmp_path / "m.gguf")
    W.write(path, [("general.architecture", W.STRING, "llama")], [W.weight_tensor("blk.0.ffn_down.weight", qtype, b, N, K)])
    with g.GGUFFile(path) as f:
        blocks, qt, n, k = f.weight("blk.0.ffn_down.weight")
    assert (qt, n, k) == (qtype, N, K) and np.array_equal(blocks, b)
    x = syn.normal(syn.rng(5), (M, K), "bf16")
    y = U.guarded((M, N), torch.float32)
    nws = g.gguf_mm_workspace_size(g.GGUF_OP_GEMM, qt, n, k, M)
    ws = U.workspace(nws)
    g.gguf_mm_gemm(U.dev(blocks), qt, 0, n, k, U.dev(x, "bf16"), g.GGUF_DT_BF16, M, None, y.t, g.GGUF_DT_F32, ws.t,
                   nws, g.GGUF_PATH_FUSED)
    torch.cuda.synchronize()
    y.check("y")
    assert g.gguf_mm_check_errors() == 0
    ref = O.matmul_exact(U.act_f64(x, "bf16"), O.dequant(b, qtype, N, K))
    U.check_close(U.host64(y.t), ref, "f32", rel=2e-3, what=f"q{qtype} from file")
