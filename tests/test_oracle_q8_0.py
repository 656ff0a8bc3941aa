"""Pins for the oracle's q8_0 quantizer.

The pages name q8_0 ("07 . R3", section 1) and state that the quantizer's
amax scan is order-independent ("Lecture 08", section 8).  The rest of the
definition (fp32 d = amax/127, fp32 IEEE x/d, round half away from zero,
binary16 stored scale) is the stated reading.  These tests check properties
and hand-derived values, never a re-typed copy of the formula.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
from tests.q4k_layout import q8_fields


def _q(x):
    out = oracle.quantize_q8_0(np.asarray(x, np.float32).reshape(1, -1))
    K = np.asarray(x).size
    dq, qi = q8_fields(out, K)
    return out[0], dq[0], qi[0].reshape(-1)


def test_block_size_and_layout():
    x = np.arange(64, dtype=np.float32) - 20
    raw, dq, qi = _q(x)
    assert raw.size == 68
    # the stored scale is little-endian binary16 at bytes 0-1 of each block
    for b in range(2):
        bits = int(raw[34 * b]) | (int(raw[34 * b + 1]) << 8)
        assert np.uint16(bits).view(np.float16) == np.float16(dq[b])


def test_ties_round_half_away_from_zero():
    # amax = 127 makes d = 1 exactly, so x/d = x and every .5 is a tie
    x = np.zeros(32, np.float32)
    x[0] = 127.0
    x[1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, -126.5]
    x[9:13] = [3.0, -3.0, 0.49999997, -0.49999997]
    raw, dq, qi = _q(x)
    assert dq[0] == 1.0
    assert list(qi[:13]) == [127, 3, -3, 1, -1, 2, -2, 127, -127, 3, -3, 0, 0]


def test_integer_inputs_are_exact():
    x = np.arange(-16, 16, dtype=np.float32)
    x[0] = -127.0
    raw, dq, qi = _q(x)
    assert dq[0] == 1.0
    assert np.array_equal(qi, x.astype(np.int64))


def test_zero_block():
    raw, dq, qi = _q(np.zeros(32, np.float32))
    assert np.all(raw == 0)


def test_max_magnitude_maps_to_127_and_signs():
    rng = np.random.default_rng(7)
    for _ in range(200):
        x = rng.standard_normal(32).astype(np.float32) * np.float32(10 ** rng.uniform(-3, 3))
        raw, dq, qi = _q(x)
        i = int(np.argmax(np.abs(x)))
        assert abs(qi[i]) == 127 and np.sign(qi[i]) == np.sign(x[i])
        assert np.all(np.abs(qi) <= 127)
        assert np.all((qi == 0) | (np.sign(qi) == np.sign(x)))


def test_scale_is_binary16_of_fp32_quotient():
    rng = np.random.default_rng(8)
    x = (rng.standard_normal((50, 32)) * 3).astype(np.float32)
    out = oracle.quantize_q8_0(x.reshape(1, -1))
    dq, qi = q8_fields(out, x.size)
    amax = np.abs(x).max(axis=1)
    d32 = amax / np.float32(127.0)                    # numpy: IEEE fp32 division
    assert d32.dtype == np.float32
    assert np.array_equal(dq[0].astype(np.float16).view(np.uint16), d32.astype(np.float16).view(np.uint16))


def test_reconstruction_error_bound():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((64, 32)) * np.float32(2.0)).astype(np.float32)
    x[5, 3] *= 20
    out = oracle.quantize_q8_0(x.reshape(1, -1))
    dq, qi = q8_fields(out, x.size)
    amax = np.abs(x).max(axis=1).astype(np.float64)
    d_exact = amax / 127.0
    # quantization used the fp32 quotient; the stored scale adds binary16 rounding on top
    rec = dq[0][:, None] * qi[0]
    bound = d_exact[:, None] * (0.5 + 1e-6) + 127.0 * np.abs(dq[0] - d_exact)[:, None]
    assert np.all(np.abs(rec - x.astype(np.float64)) <= bound)


def test_order_independence_of_scale():
    # the amax scan is a max over magnitudes: permuting a block permutes q, keeps d
    rng = np.random.default_rng(10)
    x = rng.standard_normal(32).astype(np.float32)
    raw, dq, qi = _q(x)
    for _ in range(20):
        p = rng.permutation(32)
        raw2, dq2, qi2 = _q(x[p])
        assert raw2[0] == raw[0] and raw2[1] == raw[1]
        assert np.array_equal(qi2, qi[p])


def test_blocks_are_independent():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(96).astype(np.float32)
    whole = oracle.quantize_q8_0(x.reshape(1, -1))[0]
    parts = np.concatenate([oracle.quantize_q8_0(x[32 * b:32 * b + 32].reshape(1, -1))[0] for b in range(3)])
    assert np.array_equal(whole, parts)


def _half_away(fr: Fraction) -> int:
    # exact round half away from zero of a rational
    n = abs(fr)
    k = math.floor(n + Fraction(1, 2))
    return k if fr >= 0 else -k


def test_hand_worked_block():
    # x_i = i - 15.5: amax = 15.5, d = 15.5/127, q_i = round(x_i * 127 / 15.5).
    # The exact rational quotient is at least 1e-3 away from every .5 tie, so the
    # fp32 division the definition uses cannot move any of them across a tie.
    x = np.arange(32, dtype=np.float32) - np.float32(15.5)
    expect = []
    for i in range(32):
        v = Fraction(2 * i - 31, 2) * 127 / Fraction(31, 2)
        frac = abs(v) - math.floor(abs(v))
        assert abs(frac - Fraction(1, 2)) > Fraction(1, 1000)
        expect.append(_half_away(v))
    raw, dq, qi = _q(x)
    assert list(qi) == expect
    assert expect[0] == -127 and expect[31] == 127
    assert np.float16(dq[0]) == np.float16(np.float32(15.5) / np.float32(127))


def test_multi_column_independent():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((3, 64)).astype(np.float32)
    allc = oracle.quantize_q8_0(x)
    for c in range(3):
        assert np.array_equal(allc[c], oracle.quantize_q8_0(x[c:c + 1])[0])


def _find_div_vs_recip_case():
    # search, with numpy's IEEE fp32 arithmetic, for a value whose code differs
    # between x/d and x*(1/d) (both rounded half away from zero): the reading
    # fixes division
    rng = np.random.default_rng(13)
    one = np.float32(1.0)
    for _ in range(2000):
        amax = np.float32(rng.uniform(0.5, 100.0))
        d = amax / np.float32(127.0)
        k = rng.integers(1, 126)
        base = (np.float32(k) + np.float32(0.5)) * d
        for direction in (np.float32(np.inf), np.float32(-np.inf)):
            x = np.float32(base)
            for _s in range(8):
                qa = _half_away(Fraction(float(x / d)))
                qb = _half_away(Fraction(float(x * (one / d))))
                if qa != qb:
                    return amax, x, qa, qb
                x = np.nextafter(x, direction)
    return None


def test_division_not_reciprocal_multiply():
    found = _find_div_vs_recip_case()
    assert found is not None
    amax, x, q_div, q_rec = found
    blk = np.zeros(32, np.float32)
    blk[0] = amax
    blk[1] = x
    raw, dq, qi = _q(blk)
    assert qi[0] == 127
    assert qi[1] == q_div and qi[1] != q_rec
