"""Pins of the fp8 (E4M3) oracle against facts of the format and of scaling that do
not come from the oracle's own code: hand-derived representable values, rounding
ties, saturation, and exact closed forms of the scaled products."""
import numpy as np
import pytest

from oracle import fp8_oracle as F8

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_grid_matches_the_format_by_hand():
    g = F8.e4m3_grid()
    assert len(g) == 127                       # 8 subnormals (with 0) + 14 x 8 + 7 normals
    assert g[0] == 0.0 and g[1] == 2.0 ** -9   # smallest subnormal: 1/8 * 2^-6
    assert g[-1] == 448.0 and g[-2] == 416.0   # 1.75 * 2^8, 1.625 * 2^8
    one = np.searchsorted(g, 1.0)
    assert list(g[one:one + 8]) == [1.0, 1.125, 1.25, 1.375, 1.5, 1.625, 1.75, 1.875]
    assert 2.0 ** -6 in g and 7 / 8 * 2.0 ** -6 in g   # smallest normal, largest subnormal


def test_representable_values_round_trip_with_either_sign():
    g = F8.e4m3_grid()
    assert np.array_equal(F8.quantize_e4m3(g), g)
    assert np.array_equal(F8.quantize_e4m3(-g), -g)


@pytest.mark.parametrize("v,want", [
    (1.0625, 1.0),            # tie between 1 (m=0) and 1.125 (m=1): even
    (1.1875, 1.25),           # tie between 1.125 (m=1) and 1.25 (m=2): even
    (1.06, 1.0), (1.07, 1.125),
    (-3.1, -3.0),             # 3.0 = 1.5 * 2, 3.25 = 1.625 * 2
    (232.0, 224.0),           # tie between 224 (m=6) and 240 (m=7): even
    (236.0, 240.0),
    (464.0, 448.0), (500.0, 448.0), (-1e9, -448.0),   # saturation
    (2.0 ** -10, 0.0),        # half the smallest subnormal: tie with 0, even
    (3 * 2.0 ** -10, 2.0 ** -8),   # tie between 2^-9 (m=1) and 2^-8 (m=2): even
    (0.0, 0.0),
])
def test_rounding_cases(v, want):
    assert F8.quantize_e4m3(np.array([v]))[0] == want


def test_nan_stays_nan():
    assert np.isnan(F8.quantize_e4m3(np.array([np.nan]))[0])


def test_row_scaling_maps_each_row_max_to_448():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((5, 77)).astype(np.float32)
    w[2] = 0.0
    q, s = F8.quantize_rows(w)
    assert s.dtype == np.float32 and s[2] == 1.0
    for r in (0, 1, 3, 4):
        assert np.max(np.abs(q[r])) == 448.0
    assert np.all(q[2] == 0.0)
    # every code is a representable value
    g = F8.e4m3_grid()
    assert np.all(np.isin(np.abs(q), g))


def test_gemv_exact_when_everything_is_representable():
    # rows and tokens whose largest magnitude is 448 have scale 1: codes equal the
    # values, so y is the plain product
    rng = np.random.default_rng(5)
    g = F8.e4m3_grid()
    w = rng.choice(g, size=(6, 64)) * rng.choice([-1.0, 1.0], size=(6, 64))
    x = rng.choice(g, size=(3, 64)) * rng.choice([-1.0, 1.0], size=(3, 64))
    w[:, 0] = 448.0
    x[:, 5] = -448.0
    wq, ws = F8.quantize_rows(w)
    assert np.all(ws == 1.0) and np.array_equal(wq, w)
    y = F8.gemv_e4m3(wq, ws, x)
    assert np.array_equal(y, x @ w.T)


def test_gemv_scales_by_powers_of_two_exactly():
    rng = np.random.default_rng(7)
    w = rng.standard_normal((9, 128)).astype(np.float32)
    x = rng.standard_normal((4, 128)).astype(np.float32)
    wq, ws = F8.quantize_rows(w)
    y = F8.gemv_e4m3(wq, ws, x)
    wq2, ws2 = F8.quantize_rows(w * np.float32(8.0))
    x2 = x * np.float32(0.25)
    assert np.array_equal(wq2, wq) and np.array_equal(ws2, ws * np.float32(8.0))
    assert np.allclose(F8.gemv_e4m3(wq2, ws2, x2), 2.0 * y, rtol=0, atol=0)


def test_gemv_close_to_the_unquantised_product():
    # Each code is within 1/16 relative of its value (3 mantissa bits), a rounding
    # error of standard deviation at most (1/16)/sqrt(3) = 3.6%; with both factors
    # rounded independently and 1280 terms of random sign, the RMS error of y is at
    # most sqrt(2) * 3.6% = 5.1% of y's RMS.
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((256, 1280)) / np.sqrt(1280)).astype(np.float32)
    x = rng.standard_normal((8, 1280)).astype(np.float32)
    wq, ws = F8.quantize_rows(w)
    y = F8.gemv_e4m3(wq, ws, x)
    ref = x.astype(np.float64) @ w.T.astype(np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.sqrt(np.mean((y - ref) ** 2)) / rms < 0.051
    assert np.sqrt(np.mean((y - ref) ** 2)) / rms > 0.005   # it is quantised at all
