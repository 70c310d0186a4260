"""Pins of the oracle's MXFP8 quantisation (``oracle/mx.py``) to the format's
definition (CPU only):

* the 256 E4M3 codes decode to 254 distinct-sign finite values and two NaNs,
  the extremes are 448 and the 2^-9 subnormal, and every finite value is a
  fixed point of the rounding (the decoder reads bit fields, the rounding
  works on value spacings: two independent statements of the format);
* between neighbouring values, points just off the midpoint round to the
  nearer one and the midpoint itself to the code with the even mantissa;
* magnitudes past 448 clamp; block exponents follow floor(log2 max|x|) - 8,
  including the clamp of a block maximum in (448, 512) and all-zero blocks;
* the round trip of normal-range elements is within half a unit in the last
  place (2^-4 relative), of subnormal ones within 2^-10 of the block scale.
"""

import numpy as np
import pytest

from oracle import mx


def _finite_codes():
    vals = [(c, mx.e4m3_value(c)) for c in range(256)]
    return [(c, v) for c, v in vals if not np.isnan(v)]


def test_code_table():
    vals = [mx.e4m3_value(c) for c in range(256)]
    assert sum(np.isnan(v) for v in vals) == 2
    fin = [v for v in vals if not np.isnan(v)]
    assert len(fin) == 254
    assert max(fin) == 448.0 and min(fin) == -448.0
    pos = sorted({v for v in fin if v > 0})
    assert pos[0] == 2.0 ** -9 and len(pos) == 126
    assert mx.e4m3_value(0x38) == 1.0          # exponent field 7 = bias
    assert mx.e4m3_value(0x08) == 2.0 ** -6    # smallest normal


def test_every_value_is_a_fixed_point():
    for _, v in _finite_codes():
        assert mx.round_e4m3(v) == v


def test_nearest_and_ties_to_even():
    pos = sorted({(v, c) for c, v in _finite_codes() if v >= 0})
    for (a, ca), (b, cb) in zip(pos, pos[1:]):
        mid = (a + b) / 2
        eps = (b - a) * 1e-6
        assert mx.round_e4m3(mid - eps) == a
        assert mx.round_e4m3(mid + eps) == b
        even = a if (ca & 1) == 0 else b
        assert mx.round_e4m3(mid) == even
        assert mx.round_e4m3(-mid) == -even


def test_clamp():
    assert mx.round_e4m3(448.0) == 448.0
    assert mx.round_e4m3(463.9) == 448.0
    assert mx.round_e4m3(1e9) == 448.0
    assert mx.round_e4m3(-1e9) == -448.0


def test_block_exponents_and_scaled_elements():
    x = np.zeros((3, 64))
    x[0, :32] = np.linspace(-1.0, 1.0, 32)        # max 1   -> 2^(0 - 8)
    x[0, 32:] = 500.0                             # max 500 -> 2^(8 - 8), clamps
    x[1, 5] = -3.0                                # max 3   -> 2^(1 - 8)
    el, ex = mx.quantise(x)
    assert ex.tolist() == [[-8, 0], [-7, -127], [-127, -127]]
    assert np.all(el[0, 32:] == 448.0)
    assert el[0, 31] == 256.0 and el[0, 0] == -256.0
    assert el[1, 5] == -3.0 * 2 ** 7 == mx.round_e4m3(-384.0)
    assert not el[2].any() and not el[1, 32:].any()


@pytest.mark.parametrize("seed", range(3))
def test_round_trip_error_bound(seed):
    g = np.random.default_rng(seed)
    x = g.standard_normal((64, 128)) * np.exp(g.uniform(-8, 8, size=(64, 1)))
    x[:, 7] *= 1e-6                               # deep subnormals inside a block
    el, ex = mx.quantise(x)
    rt = mx.dequantise(el, ex)
    scale = np.repeat(2.0 ** ex.astype(np.float64), 32, axis=-1)
    mag = np.abs(x) / scale
    ok = mag <= 448.0                             # not clipped
    normal = ok & (mag >= 2.0 ** -6)
    sub = ok & (mag < 2.0 ** -6)
    err = np.abs(x - rt)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]) * (1 + 1e-12))
    assert np.all(err[sub] <= 2.0 ** -10 * scale[sub] * (1 + 1e-12))
    assert np.array_equal(mx.mx_round_trip(x), rt)
