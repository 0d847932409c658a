"""Pins for the oracle's KV helpers (CPU only): widening, the INT8/INT4 codecs,
the scale layout, page-table expansion and row appends.

The codecs are checked with exact rational arithmetic (``fractions``) and
hand-worked cases rather than by re-running their own numpy steps.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth


def test_widening_is_exact_for_known_bit_patterns():
    assert oracle.widen_bf16(np.array([0x3F80], np.uint16))[0] == 1.0
    assert oracle.widen_bf16(np.array([0xC040], np.uint16))[0] == -3.0
    assert oracle.widen_bf16(np.array([0x3F81], np.uint16))[0] == 1.0 + 2.0 ** -7
    assert oracle.widen_f16(np.array([0x3C00], np.uint16))[0] == 1.0
    assert oracle.widen_f16(np.array([0x0001], np.uint16))[0] == 2.0 ** -24
    assert oracle.widen_f16(np.array([0x7BFF], np.uint16))[0] == 65504.0


def _fp16_neighbours(x: float):
    h = np.float16(x)
    return float(np.nextafter(h, np.float16(-np.inf))), float(h), float(np.nextafter(h, np.float16(np.inf)))


# --- INT8 ---------------------------------------------------------------------


def test_int8_round_trip_is_exact_on_the_grid():
    g = np.random.default_rng(1)
    N, H, D = 40, 3, 64
    s = g.uniform(0.001, 3.0, size=(N, H)).astype(np.float16)
    q = g.integers(-127, 128, size=(N, H, D))
    q[:, :, 5] = np.where(g.random((N, H)) < 0.5, 127, -127)      # amax code is +-127
    x = q.astype(np.float32) * s.astype(np.float32)[..., None]   # exact products
    q2, s2 = oracle.quantize_int8(x)
    np.testing.assert_array_equal(s2, s)
    np.testing.assert_array_equal(q2, q.astype(np.int8))
    np.testing.assert_array_equal(oracle.dequantize_int8(q2, s2), x)


def test_int8_scale_is_nearest_fp16_of_amax_over_127():
    g = np.random.default_rng(2)
    x = oracle.widen_bf16(synth.normal_bits(synth.rng(7), (64, 4, 32), "bf16"))
    _, s = oracle.quantize_int8(x)
    amax = np.abs(x).max(axis=-1)
    for a, got in zip(amax.ravel(), s.ravel()):
        exact = Fraction(float(a)) / 127
        lo, mid, hi = _fp16_neighbours(float(got))
        # got is at least as close to the exact ratio as either fp16 neighbour
        # (the intermediate fp32 rounding can only matter at exact fp16 ties)
        d = abs(Fraction(mid) - exact)
        assert d <= abs(Fraction(lo) - exact) and d <= abs(Fraction(hi) - exact)


def test_int8_codes_are_nearest_integers_ties_to_even():
    x = oracle.widen_bf16(synth.normal_bits(synth.rng(8), (128, 2, 64), "bf16"))
    q, s = oracle.quantize_int8(x)
    for r in range(x.shape[0]):
        for h in range(x.shape[1]):
            sf = Fraction(float(s[r, h]))
            for d in range(x.shape[2]):
                t = Fraction(float(x[r, h, d])) / sf
                c = int(q[r, h, d])
                if abs(t) > 127:
                    assert c == (127 if t > 0 else -127)
                    continue
                err = abs(t - c)
                assert err <= Fraction(1, 2) + Fraction(1, 1 << 20)
                if err == Fraction(1, 2):
                    assert c % 2 == 0


def test_int8_ties_round_to_even_exact_cases():
    s = np.float16(0.5)
    row = np.zeros((1, 1, 8), np.float32)
    row[0, 0, :] = [2.5 * 0.5, 3.5 * 0.5, -2.5 * 0.5, -3.5 * 0.5, 0.5 * 0.5, 1.5 * 0.5, 0.0, 127 * 0.5]
    q, s2 = oracle.quantize_int8(row)
    assert s2[0, 0] == s
    assert q[0, 0].tolist() == [2, 4, -2, -4, 0, 2, 0, 127]


def test_int8_zero_row_and_saturated_scale():
    z = np.zeros((1, 2, 16), np.float32)
    z[0, 1, 3] = 3.0e38          # a bf16-representable huge value: amax/127 overflows fp16
    q, s = oracle.quantize_int8(z)
    assert s[0, 0] == 0 and np.all(q[0, 0] == 0)
    assert float(s[0, 1]) == 65504.0 and q[0, 1, 3] == 127


def _rows_with_non_finite():
    """Rows [NaN row, +Inf row, -Inf row, finite row], one head, D = 8."""
    x = np.array([[1.0, 2.0, np.nan, -3.0, 0.5, 0.0, 4.0, -1.0],
                  [1.0, np.inf, -2.0, 0.25, 0.0, 3.0, -1.0, 2.0],
                  [-np.inf, 1.0, 2.0, 3.0, 4.0, 5.0, 6.0, 7.0],
                  [127.0, -63.5, 0.0, 1.0, 2.0, -2.0, 63.5, -127.0]], np.float32)
    return x[:, None, :]


def test_int8_non_finite_rows():
    # the non-finite reading: a NaN row keeps its NaN (scale 0x7E00, every
    # code 0, so every dequantised value is NaN); an Inf element makes
    # amax/127 = Inf, clamped to the largest fp16 65504, and codes as +-127
    # while the finite elements of its row (|x| <= 7 here) round to 0
    q, s = oracle.quantize_int8(_rows_with_non_finite())
    bits = s.view(np.uint16)[:, 0].tolist()
    assert bits[0] == 0x7E00 and q[0, 0].tolist() == [0] * 8
    assert np.isnan(oracle.dequantize_int8(q, s)[0]).all()
    assert bits[1] == 0x7BFF and q[1, 0].tolist() == [0, 127, 0, 0, 0, 0, 0, 0]
    assert bits[2] == 0x7BFF and q[2, 0].tolist() == [-127, 0, 0, 0, 0, 0, 0, 0]
    # the finite row is untouched by its neighbours: scale 1.0 exactly (0x3C00), ties to even
    assert bits[3] == 0x3C00 and q[3, 0].tolist() == [127, -64, 0, 1, 2, -2, 64, -127]


def test_int4_non_finite_rows():
    packed, s = oracle.quantize_int4(_rows_with_non_finite())
    bits = s.view(np.uint16)[:, 0].tolist()
    assert bits[0] == 0x7E00 and packed[0, 0].tolist() == [0, 0, 0, 0]
    assert np.isnan(oracle.dequantize_int4(packed, s)[0]).all()
    # +Inf -> code 7 in the high nibble of byte 0; -Inf -> code -7 (0x9) in the low nibble
    assert bits[1] == 0x7BFF and packed[1, 0].tolist() == [0x70, 0, 0, 0]
    assert bits[2] == 0x7BFF and packed[2, 0].tolist() == [0x09, 0, 0, 0]


def test_int8_dequantisation_is_the_exact_product():
    g = np.random.default_rng(3)
    q = g.integers(-127, 128, size=(10, 2, 8)).astype(np.int8)
    s = g.uniform(1e-4, 100, size=(10, 2)).astype(np.float16)
    x = oracle.dequantize_int8(q, s)
    for idx in np.ndindex(q.shape):
        assert Fraction(float(x[idx])) == Fraction(int(q[idx])) * Fraction(float(s[idx[:2]]))


def test_scale_layout_is_page_major_then_head_then_offset():
    R, H = 128, 2
    s = np.array([[r * 10 + g for g in range(H)] for r in range(R)], dtype=np.float16)
    sp = oracle.pack_scales(s)
    assert sp.shape == (2, 2, 64)
    assert sp[1, 1, 3] == s[67, 1] and sp[0, 0, 63] == s[63, 0] and sp[1, 0, 0] == s[64, 0]
    np.testing.assert_array_equal(oracle.unpack_scales(sp), s)


# --- INT4 ---------------------------------------------------------------------


def test_int4_round_trip_on_grid_and_nibble_order():
    s = np.array([[0.25]], np.float16)
    codes = np.array([[[7, -7, 1, -1, 0, 3, -4, 6]]])
    x = codes.astype(np.float32) * np.float32(0.25)
    packed, s2 = oracle.quantize_int4(x)
    assert s2[0, 0] == s[0, 0]
    # element 2t in the low nibble, 2t+1 in the high nibble, two's complement
    assert packed[0, 0].tolist() == [0x97, 0xF1, 0x30, 0x6C]
    np.testing.assert_array_equal(oracle.dequantize_int4(packed, s2), x)


def test_int4_codes_are_nearest_with_ties_to_even():
    x = oracle.widen_bf16(synth.normal_bits(synth.rng(9), (32, 2, 16), "bf16"))
    packed, s = oracle.quantize_int4(x)
    deq = oracle.dequantize_int4(packed, s)
    for idx in np.ndindex(x.shape):
        sf = Fraction(float(s[idx[:2]]))
        t = Fraction(float(x[idx])) / sf
        c = Fraction(float(deq[idx])) / sf
        if abs(t) > 7:
            assert abs(c) == 7
            continue
        assert abs(t - c) <= Fraction(1, 2) + Fraction(1, 1 << 20)
        if abs(t - c) == Fraction(1, 2):
            assert c.numerator % 2 == 0


# --- page tables ----------------------------------------------------------------


def test_page_table_expansion_hand_worked():
    pt = np.array([[2, 0, -1], [1, -1, -1]], dtype=np.int32)
    rows = oracle.page_table_to_rows(pt, np.array([70, 5]), 130, page=64)
    want0 = list(range(128, 192)) + list(range(0, 6)) + [-1] * 60
    want1 = list(range(64, 69)) + [-1] * 125
    assert rows[0].tolist() == want0
    assert rows[1].tolist() == want1


def test_negative_page_ids_and_overlong_lengths_are_padding():
    pt = np.array([[3, -1, 1]], dtype=np.int32)
    rows = oracle.page_table_to_rows(pt, np.array([500]), 200, page=64)
    assert rows[0, :64].tolist() == list(range(192, 256))
    assert np.all(rows[0, 64:128] == -1)
    assert rows[0, 128:192].tolist() == list(range(64, 128))
    assert np.all(rows[0, 192:] == -1)          # beyond max_pages * page


def test_identity_page_table_gives_contiguous_rows():
    pt = np.arange(8, dtype=np.int32)[None]
    rows = oracle.page_table_to_rows(pt, np.array([500]), 512)
    assert rows[0, :500].tolist() == list(range(500)) and np.all(rows[0, 500:] == -1)


# --- appends ---------------------------------------------------------------------


def test_append_copy_writes_named_rows_only():
    pool = np.zeros((6, 1, 2), np.uint16)
    new = np.array([[[1, 2]], [[3, 4]], [[5, 6]]], np.uint16)
    out, _ = oracle.append_rows(pool, new, np.array([4, -1, 0]))
    assert out[:, 0].tolist() == [[5, 6], [0, 0], [0, 0], [0, 0], [1, 2], [0, 0]]


def test_append_int8_matches_quantising_the_rows_in_place():
    g = np.random.default_rng(4)
    new = oracle.widen_bf16(synth.normal_bits(synth.rng(10), (3, 2, 16), "bf16"))
    pool = np.zeros((128, 2, 16), np.int8)
    sc = np.zeros((2, 2, 64), np.float16)
    out, sc2 = oracle.append_rows(pool, new, np.array([70, 3, -2]), sc, fmt="int8")
    qv, s = oracle.quantize_int8(new)
    np.testing.assert_array_equal(out[70], qv[0])
    np.testing.assert_array_equal(out[3], qv[1])
    assert sc2[1, 0, 6] == s[0, 0] and sc2[0, 1, 3] == s[1, 1]
    assert np.count_nonzero(sc2) == np.count_nonzero(s[:2])
