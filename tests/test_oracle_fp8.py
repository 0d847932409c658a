"""Pins of the oracle's FP8 E4M3 codec: the format's defining values, every
code's round trip, midpoints (ties to even), saturation and NaN, and the
quantiser's scale rule."""
import numpy as np

import oracle


def test_defining_values_of_the_format():
    v = oracle.e4m3_value
    assert v(0x00) == 0.0 and v(0x80) == 0.0 and np.signbit(v(0x80))
    assert v(0x01) == 2.0 ** -9                 # smallest subnormal
    assert v(0x07) == 7 * 2.0 ** -9             # largest subnormal
    assert v(0x08) == 2.0 ** -6                 # smallest normal
    assert v(0x38) == 1.0                       # exponent 7 = bias
    assert v(0x7E) == 448.0 and v(0xFE) == -448.0
    assert np.isnan(v(0x7F)) and np.isnan(v(0xFF))
    assert v(0x78) == 256.0 and v(0x3C) == 1.5


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle.e4m3_value(codes)
    back = oracle.e4m3_encode(vals)
    # -0 encodes as 0x80 (sign kept); all others exactly
    assert np.array_equal(back, codes)


def test_midpoints_round_to_the_even_code():
    codes = np.array([c for c in range(0x7E)], np.uint8)        # positive finite codes 0..447 (0x7E is 448)
    lo, hi = oracle.e4m3_value(codes), oracle.e4m3_value(codes + 1)
    mid = (lo + hi) / 2.0
    got = oracle.e4m3_encode(mid)
    want = np.where(codes % 2 == 0, codes, codes + 1)            # the even mantissa wins
    assert np.array_equal(got, want.astype(np.uint8))
    # just off the midpoint goes to the nearer side
    assert np.array_equal(oracle.e4m3_encode(mid * (1 - 1e-9)), codes)
    assert np.array_equal(oracle.e4m3_encode(mid * (1 + 1e-9)), (codes + 1).astype(np.uint8))


def test_saturation_and_nan():
    y = np.array([448.0, 464.0, 480.0, 1e6, np.inf, -1e30, np.nan], np.float64)
    got = oracle.e4m3_encode(y)
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F]


def test_quantiser_scale_and_exact_dequantisation():
    g = np.random.default_rng(3)
    x = g.standard_normal((50, 3, 64)).astype(np.float32)
    x[4, 1] = 0.0
    q, s = oracle.quantize_fp8(x)
    amax = np.abs(x).max(-1)
    assert np.array_equal(s, np.minimum(amax / np.float32(448), np.float32(65504)).astype(np.float16))
    assert not q[4, 1].any() and s[4, 1] == 0
    deq = oracle.dequantize_fp8(q, s)
    # exact product of the two factors
    want = (oracle.e4m3_value(q) * s.astype(np.float64)[..., None])
    assert np.array_equal(deq.astype(np.float64), want)
    # the largest element of each row maps to the top of the grid (448, or the saturated code)
    top = np.abs(oracle.e4m3_value(q)).max(-1)
    assert np.all((top[s > 0] >= 416) & (top[s > 0] <= 448))
    # relative error of a code is at most half a step: 2^-4 of the value for normals
    ok = (np.abs(x) >= s.astype(np.float32)[..., None] * 2.0 ** -6) & (np.abs(x) > 0)
    rel = np.abs(deq - x)[ok] / np.abs(x)[ok]
    assert rel.max() <= 2.0 ** -4 * 1.0001


def test_quantiser_non_finite_rows():
    # the non-finite reading: a NaN anywhere in a (row, head) gives scale
    # 0x7E00 and the NaN code 0x7f for every element; an Inf element gives
    # scale 65504 (amax/448 = Inf, clamped) and saturates to +-448 (0x7E /
    # 0xFE), while the finite elements (|x| <= 5) fall far below the
    # smallest subnormal step (2^-9 * 65504 = 128) and code as +-0
    x = np.array([[3.0, np.nan, -1.0, 2.0],
                  [1.0, np.inf, -3.0, 0.0],
                  [-np.inf, 5.0, -0.0, 1.0]], np.float32)[:, None, :]
    q, s = oracle.quantize_fp8(x)
    bits = s.view(np.uint16)[:, 0].tolist()
    assert bits == [0x7E00, 0x7BFF, 0x7BFF]
    assert q[0, 0].tolist() == [0x7F] * 4
    assert q[1, 0].tolist() == [0x00, 0x7E, 0x80, 0x00]
    assert q[2, 0].tolist() == [0xFE, 0x00, 0x80, 0x00]
    assert np.isnan(oracle.dequantize_fp8(q, s)[0]).all()
