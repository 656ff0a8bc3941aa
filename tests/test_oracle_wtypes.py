"""Pins of the oracle's q4_0 / q8_0 weight matvec (the weight types of the pages'
other models, against q8_0 activations), each against something other than the
oracle's own formula: hand-built blocks with known values, an independent numpy
unpack, exact rational arithmetic, and special cases."""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth

F16_ONE = (0x00, 0x3C)


def _q4_0_block(d_bits: int, nibbles):
    """18-byte block from 32 nibble values (weight i -> byte i % 16, low nibble for i < 16)."""
    b = np.zeros(18, np.uint8)
    b[0], b[1] = d_bits & 0xFF, d_bits >> 8
    for i in range(16):
        b[2 + i] = (nibbles[i] & 15) | ((nibbles[i + 16] & 15) << 4)
    return b


def _np_dequant(wtype, row, K):
    """independent numpy unpack of a q4_0 / q8_0 row"""
    bb = oracle.W_BLOCK_BYTES[wtype]
    blk = row.reshape(K // 32, bb)
    d = blk[:, 0:2].copy().view(np.float16).astype(np.float64).reshape(-1, 1)
    if wtype == "q4_0":
        lo = (blk[:, 2:18] & 15).astype(np.int64) - 8
        hi = (blk[:, 2:18] >> 4).astype(np.int64) - 8
        q = np.concatenate([lo, hi], axis=1)
    else:
        q = blk[:, 2:34].copy().view(np.int8).astype(np.int64)
    return (d * q).reshape(-1)


def test_q4_0_closed_form_all_equal():
    # every nibble q and scale d: every weight is d*(q-8), exactly
    for q in (0, 1, 7, 8, 9, 15):
        for d_bits in (0x3C00, 0x2E66, 0x0001, 0x7BFF):
            blk = _q4_0_block(d_bits, [q] * 32)
            w = oracle.dequant_w_row("q4_0", np.tile(blk, 8), 256)
            d = float(np.array([d_bits], np.uint16).view(np.float16)[0])
            assert np.all(w == d * (q - 8))


@pytest.mark.parametrize("pos", range(32))
def test_q4_0_nibble_placement(pos):
    # all weights zero (q = 8) except one nibble set to 9: exactly weight `pos` is +d
    nib = [8] * 32
    nib[pos] = 9
    blk = _q4_0_block(0x3C00, nib)
    w = oracle.dequant_w_row("q4_0", np.tile(blk, 8), 256)
    expect = np.zeros(256)
    expect[pos::32] = 1.0
    assert np.array_equal(w, expect)


def test_q8_0_weights_match_numpy_view():
    W = synth.wq_matrix("q8_0", 3, 512, seed=5)
    for r in range(3):
        assert np.array_equal(oracle.dequant_w_row("q8_0", W[r], 512), _np_dequant("q8_0", W[r], 512))


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0"])
def test_matvec_matches_dequant_dot(wtype):
    rows, K = 7, 1024
    W = synth.wq_matrix(wtype, rows, K, seed=6)
    x = synth.activation(K, 2, seed=6)
    xq = oracle.quantize_q8_0(x)
    y, T = oracle.matvec_w(wtype, W, xq, rows, K)
    xd = oracle.dequant_q8_0(xq, K)
    for r in range(rows):
        wd = _np_dequant(wtype, W[r], K)
        ref = xd @ wd
        assert np.all(np.abs(y[:, r] - ref) <= 1e-12 * T[:, r] + 1e-300)


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0"])
def test_matvec_exact_rational_k256(wtype):
    W = synth.wq_matrix(wtype, 2, 256, seed=7)
    x = synth.activation(256, 1, seed=7)
    xq = oracle.quantize_q8_0(x)[0]
    y, _ = oracle.matvec_w(wtype, W, xq, 2, 256)
    bb = oracle.W_BLOCK_BYTES[wtype]
    for r in range(2):
        acc = Fraction(0)
        for b in range(8):
            wblk = W[r, b * bb:(b + 1) * bb]
            dw = Fraction(float(wblk[0:2].copy().view(np.float16)[0]))
            ablk = xq[b * 34:(b + 1) * 34]
            da = Fraction(float(ablk[0:2].copy().view(np.float16)[0]))
            qa = ablk[2:].view(np.int8).astype(int)
            if wtype == "q4_0":
                qw = [int(wblk[2 + (i % 16)] >> (4 * (i // 16)) & 15) - 8 for i in range(32)]
            else:
                qw = wblk[2:].view(np.int8).astype(int).tolist()
            acc += da * dw * sum(a * w for a, w in zip(qa.tolist(), qw))
        assert abs(Fraction(y[0, r]) - acc) <= abs(acc) * Fraction(1, 2 ** 40) + Fraction(1, 2 ** 80)


def test_special_cases():
    K = 256
    xq = oracle.quantize_q8_0(synth.activation(K, 1, seed=8))
    # q4_0 with every nibble 8: all weights zero
    W = np.tile(_q4_0_block(0x3C00, [8] * 32), 8).reshape(1, -1)
    y, T = oracle.matvec_w("q4_0", W, xq, 1, K)
    assert y[0, 0] == 0.0 and T[0, 0] == 0.0
    # zero activation
    xz = oracle.quantize_q8_0(np.zeros((1, K), np.float32))
    W8 = synth.wq_matrix("q8_0", 2, K, seed=8)
    y, _ = oracle.matvec_w("q8_0", W8, xz, 2, K)
    assert np.all(y == 0.0)
    # sign: q4_0 nibble 0 is -8*d
    W = np.tile(_q4_0_block(0x3C00, [0] + [8] * 31), 8).reshape(1, -1)
    assert oracle.dequant_w_row("q4_0", W[0], K)[0] == -8.0


def test_row_subset_matches_full():
    rows, K = 9, 512
    W = synth.wq_matrix("q4_0", rows, K, seed=9)
    xq = oracle.quantize_q8_0(synth.activation(K, 3, seed=9))
    y, T = oracle.matvec_w("q4_0", W, xq, rows, K)
    ids = np.array([8, 0, 4])
    ys, Ts = oracle.matvec_w("q4_0", W, xq, rows, K, row_ids=ids)
    assert np.array_equal(ys, y[:, ids]) and np.array_equal(Ts, T[:, ids])
