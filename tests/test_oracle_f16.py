"""Pins for the oracle's binary16 conversions, against numpy's IEEE float16."""
import numpy as np
import pytest

import oracle


def test_f16_to_f32_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_to_f32(int(b)) for b in bits], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))  # signed zeros too


def test_f32_to_f16_roundtrip_all_finite():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float32)
    for b, v in zip(bits, vals):
        if np.isnan(v):
            assert (oracle.f32_to_f16(float(v)) & 0x7FFF) > 0x7C00
            continue
        assert oracle.f32_to_f16(float(v)) == int(b)


def _numpy_f16_bits(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def test_f32_to_f16_ties_go_to_even():
    # midpoints between consecutive binary16 values, in the normal and subnormal ranges
    lo = np.arange(0, 0x7BFF, 7, dtype=np.uint16)
    a = lo.view(np.float16).astype(np.float64)
    b = (lo + 1).view(np.float16).astype(np.float64)
    mid = ((a + b) / 2).astype(np.float32)        # exact: fits in float32
    assert np.all(mid.astype(np.float64) == (a + b) / 2)
    ref = _numpy_f16_bits(mid)
    got = np.array([oracle.f32_to_f16(float(v)) for v in mid], dtype=np.uint16)
    assert np.array_equal(got, ref)
    # the tie goes to the neighbour with an even fraction
    assert np.all(got % 2 == 0)


def test_f32_to_f16_boundaries_and_random():
    special = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e9, -1e9, np.inf, -np.inf,
                        2.0 ** -14, 2.0 ** -14 * (1 - 2 ** -12), 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0001,
                        2.0 ** -26, 1.0, -1.0, 1.0 + 2 ** -11, 1.0 + 3 * 2 ** -11, 3.0e-5, 127.0],
                       dtype=np.float32)
    rng = np.random.default_rng(123)
    rand = np.concatenate([
        (rng.standard_normal(4000) * 10.0 ** rng.uniform(-9, 5, 4000)).astype(np.float32),
        rng.uniform(-70000, 70000, 500).astype(np.float32),
        np.abs(rng.standard_normal(2000) * 2e-3).astype(np.float32),
    ])
    vals = np.concatenate([special, rand])
    ref = _numpy_f16_bits(vals)
    got = np.array([oracle.f32_to_f16(float(v)) for v in vals], dtype=np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


def test_f32_to_f16_nan():
    assert (oracle.f32_to_f16(float("nan")) & 0x7C00) == 0x7C00
    assert (oracle.f32_to_f16(float("nan")) & 0x03FF) != 0
