"""The tolerance helper itself (CPU): the rounding interval of a bf16 / f16
value must contain every real that rounds to it and nothing that rounds
elsewhere, so the GPU tests grant exactly the final rounding."""
import numpy as np
import pytest

from tests import gpu_util as U
from oracle import gguf_oracle as O


def _to_bf16(v):
    return O.bf16_bits_to_f64(O.round_f64_to_bf16_bits(v))


def _to_f16(v):
    return np.asarray(v, np.float64).astype(np.float16).astype(np.float64)


@pytest.mark.parametrize("dtype,rnd", [("bf16", _to_bf16), ("f16", _to_f16)])
def test_rounding_interval_contains_exactly_what_rounds_to_it(dtype, rnd):
    rs = np.random.default_rng(5)
    v = np.concatenate([rs.standard_normal(20000) * 10.0 ** rs.integers(-6, 4, 20000),
                        [1.0, -1.0, 2.0, 0.5, 3.0, -4.0, 0.0]])
    got = rnd(v)
    lo, hi = U._rounding_interval(got, dtype)
    assert np.all(lo <= v) and np.all(v <= hi)
    # points just outside the interval round to a different value
    out_lo = lo - np.abs(lo) * 1e-9 - 1e-300
    out_hi = hi + np.abs(hi) * 1e-9 + 1e-300
    nz = got != 0
    assert np.all(rnd(out_lo[nz]) != got[nz]) and np.all(rnd(out_hi[nz]) != got[nz])


def test_check_close_rejects_an_error_just_above_the_bound():
    ref = np.linspace(-3, 3, 97)
    got = _to_bf16(ref)
    U.check_close(got, ref, "bf16")
    bad = got.copy()
    bad[40] = _to_bf16(ref[40] + 0.02)        # 0.02 > 2e-3 * 3 plus the rounding gap
    with pytest.raises(AssertionError):
        U.check_close(bad, ref, "bf16")
    with pytest.raises(AssertionError):
        U.check_close(ref + 3.1e-4 * 3, ref, "f32")   # raw bound for f32: 1e-4 * max|ref|
