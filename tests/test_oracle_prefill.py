"""Pins of the oracle's prefill functions ("07 . R3 -- Small-model per-token
overhead", section 1: a half-precision GEMM over a resident f16 copy of the
quantized weights).

* binary64 -> binary16 rounding against numpy's float16 conversion (a
  correctly rounded library routine), on random values of every magnitude, on
  the exact midpoints between neighbouring binary16 values (ties to even), on
  values one binary64 step either side of them, in the subnormal range and at
  the overflow boundary;
* the f16 weight cache against numpy's rounding of the oracle's binary64
  dequantization (itself pinned in test_oracle_q4K.py), and a closed form;
* the GEMM against numpy's binary64 matmul of the same binary16 values.
"""
from fractions import Fraction

import numpy as np

import oracle
from quantized_decode_matvec_gb300 import synth


def _np_f16(x):
    with np.errstate(over="ignore"):
        return np.asarray(x, np.float64).astype(np.float16).view(np.uint16)


def test_f64_to_f16_random_magnitudes():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200000) * np.exp2(rng.uniform(-30, 18, 200000))
    assert np.array_equal(oracle.f64_to_f16(x), _np_f16(x))


def test_f64_to_f16_midpoints_ties_to_even():
    # every pair of neighbouring finite binary16 values: the midpoint (exact in
    # binary64) goes to the neighbour with an even last bit; one binary64 step
    # off the midpoint goes to the nearer neighbour
    bits = np.arange(0, 0x7BFF, dtype=np.uint16)          # 0 .. the largest finite but one
    lo = bits.view(np.float16).astype(np.float64)
    hi = (bits + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2
    expect = np.where(bits % 2 == 0, bits, bits + 1).astype(np.uint16)
    assert np.array_equal(oracle.f64_to_f16(mid), expect)
    assert np.array_equal(oracle.f64_to_f16(-mid), expect | 0x8000)
    assert np.array_equal(oracle.f64_to_f16(np.nextafter(mid, 0)), bits)
    assert np.array_equal(oracle.f64_to_f16(np.nextafter(mid, np.inf)), (bits + 1).astype(np.uint16))


def test_f64_to_f16_boundaries():
    x = np.array([0.0, -0.0, 65504.0, 65519.999999, 65520.0, 1e10, np.inf, -np.inf,
                  2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25, 1e-300])
    assert np.array_equal(oracle.f64_to_f16(x), _np_f16(x))
    assert oracle.f64_to_f16(np.array([np.nan]))[0] & 0x7C00 == 0x7C00


def test_f32_to_f16_unchanged_for_binary32_inputs():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(100000) * np.exp2(rng.uniform(-28, 17, 100000))).astype(np.float32)
    got = oracle.f32_to_f16_array(x)
    assert np.array_equal(got, _np_f16(x.astype(np.float64)))
    assert all(got[i] == oracle.f32_to_f16(float(x[i])) for i in range(50))


def test_dequant_f16_is_rounded_binary64_dequant():
    W = synth.q4K_matrix(33, 768, seed=60)
    got = oracle.dequant_q4K_f16(W, 768)
    assert np.array_equal(got, _np_f16(oracle.dequant_q4K(W, 768)))


def test_dequant_f16_closed_form():
    # every field equal: every weight is d*s*q - dmin*m, computed here in exact rationals
    d_bits, dmin_bits, s, m, q = 0x1A3F, 0x0C01, 45, 19, 11
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([d_bits], np.uint16).view(np.uint8)
    blk[2:4] = np.array([dmin_bits], np.uint16).view(np.uint8)
    # six-bit scale/min pairs: low six bits of bytes 0..7 (j < 4) and the split form (j >= 4)
    for j in range(4):
        blk[4 + j] = s | ((s >> 4) << 6)
        blk[8 + j] = m | ((m >> 4) << 6)
        blk[12 + j] = (s & 15) | ((m & 15) << 4)
    blk[16:] = q | (q << 4)
    d = Fraction(float(np.array([d_bits], np.uint16).view(np.float16)[0]))
    dmin = Fraction(float(np.array([dmin_bits], np.uint16).view(np.float16)[0]))
    exact = d * s * q - dmin * m
    want = _np_f16(float(exact))[()]
    assert float(exact) == d * s * q - dmin * m  # the value is exact in binary64
    assert (oracle.dequant_q4K_f16(blk[None, :], 256) == want).all()


def test_gemm_f16_against_numpy():
    rng = np.random.default_rng(2)
    R, K, T = 37, 320, 23
    W16 = _np_f16(rng.standard_normal((R, K)) * 0.1)
    X16 = _np_f16(rng.standard_normal((T, K)))
    y, Tm = oracle.gemm_f16(W16, X16, K)
    wf = W16.view(np.float16).astype(np.float64)
    xf = X16.view(np.float16).astype(np.float64)
    ref = xf @ wf.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(Tm, np.abs(xf) @ np.abs(wf).T, rtol=1e-12)
    # a subset of rows and tokens is the same numbers
    rows, toks = np.array([36, 0, 5]), np.array([22, 1])
    ys, Ts = oracle.gemm_f16(W16, X16, K, row_ids=rows, tok_ids=toks)
    assert np.array_equal(ys, y[np.ix_(toks, rows)])
    assert np.array_equal(Ts, Tm[np.ix_(toks, rows)])


def test_gemm_f16_one_hot():
    # X a row of the identity: Y picks one column of W exactly
    K = 64
    rng = np.random.default_rng(3)
    W16 = _np_f16(rng.standard_normal((5, K)))
    X16 = np.zeros((K, K), np.uint16)
    X16[np.arange(K), np.arange(K)] = 0x3C00   # 1.0
    y, _ = oracle.gemm_f16(W16, X16, K)
    assert np.array_equal(y, W16.view(np.float16).astype(np.float64).T)
