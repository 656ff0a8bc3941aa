"""Pins for the oracle's matvec and per-block integer sums.

Checks against: exact rational brute force at K = 256, an independent numpy
dequantize-then-dot (numpy unpack + matmul), integer sums from the independent
unpacker, and special cases whose answer is known without computing.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth
from tests.q4k_layout import dequant_q8, dequant_rows, pack_block, q8_fields, unpack_fields


def _case(rows, K, ncols=1, seed=0):
    W = synth.q4K_matrix(rows, K, seed, synth.TAG_W)
    x = synth.activation(K, ncols, seed, synth.TAG_X)
    return W, x, oracle.quantize_q8_0(x)


def test_brute_force_exact_rational_K256():
    W, x, xq = _case(6, 256, seed=21)
    y, T = oracle.matvec(W, xq, 6, 256)
    dq, qi = q8_fields(xq, 256)
    d, dmin, sc, m, q = unpack_fields(W.reshape(6, 1, 144))
    for r in range(6):
        acc = Fraction(0)
        for e in range(256):
            j = e // 32
            w = (Fraction(d[r, 0]) * int(sc[r, 0, j]) * int(q[r, 0, e]) - Fraction(dmin[r, 0]) * int(m[r, 0, j]))
            acc += w * Fraction(dq[0, j]) * int(qi[0, j, e % 32])
        assert abs(y[0, r] - float(acc)) <= 1e-12 * T[0, r] + 1e-300


@pytest.mark.parametrize("rows,K", [(7, 256), (33, 1024), (5, 3584)])
def test_matches_dequant_then_dot(rows, K):
    W, x, xq = _case(rows, K, seed=rows)
    y, T = oracle.matvec(W, xq, rows, K)
    ref = dequant_rows(W, K) @ dequant_q8(xq, K)[0]
    assert np.all(np.abs(y[0] - ref) <= 1e-12 * T[0])
    # the oracle's own dequantize agrees with the independent one bit for bit
    assert np.array_equal(oracle.dequant_q4K(W, K), dequant_rows(W, K))
    assert np.array_equal(oracle.dequant_q8_0(xq, K), dequant_q8(xq, K))


def test_T_bounds_the_terms():
    W, x, xq = _case(9, 512, seed=3)
    y, T = oracle.matvec(W, xq, 9, 512)
    assert np.all(T >= np.abs(y))
    w = dequant_rows(W, 512)
    # T collects the two products per block, so it is at least the sum of |per-block contributions|
    xd = dequant_q8(xq, 512)[0]
    per_block = (w * xd).reshape(9, 16, 32).sum(axis=2)
    assert np.all(T[0] >= np.abs(per_block).sum(axis=1) * (1 - 1e-12))


def test_block_sums_exact():
    rows, K = 11, 768
    W, x, xq = _case(rows, K, ncols=2, seed=5)
    sumi, sumq = oracle.block_sums(W, xq, rows, K)
    d, dmin, sc, m, q = unpack_fields(W.reshape(rows, K // 256, 144))
    qv = q.reshape(rows, K // 32, 32)
    dq, qi = q8_fields(xq, K)
    for c in range(2):
        assert np.array_equal(sumq[c], qi[c].sum(axis=1))
        assert np.array_equal(sumi[c], np.einsum("rjk,jk->rj", qv, qi[c]))


def test_multi_column_and_row_sampling():
    rows, K = 40, 1024
    W, x, xq = _case(rows, K, ncols=3, seed=6)
    y, T = oracle.matvec(W, xq, rows, K)
    for c in range(3):
        y1, T1 = oracle.matvec(W, xq[c:c + 1], rows, K)
        assert np.array_equal(y1[0], y[c]) and np.array_equal(T1[0], T[c])
    ids = np.array([39, 0, 17, 17, 5])
    ys, Ts = oracle.matvec(W, xq, rows, K, row_ids=ids)
    assert np.array_equal(ys, y[:, ids]) and np.array_equal(Ts, T[:, ids])


def test_zero_activation_gives_zero():
    W, _, _ = _case(8, 512)
    xq = oracle.quantize_q8_0(np.zeros((1, 512), np.float32))
    y, T = oracle.matvec(W, xq, 8, 512)
    assert np.all(y == 0) and np.all(T == 0)


def test_zero_scales_and_mins_give_zero():
    rng = np.random.default_rng(0)
    blk = pack_block(0x3C00, 0x3C00, [0] * 8, [0] * 8, rng.integers(0, 16, 256))
    W = np.tile(blk, (3, 2))  # 3 rows, K = 512
    x = synth.activation(512, 1, 1)
    y, _ = oracle.matvec(W, oracle.quantize_q8_0(x), 3, 512)
    assert np.all(y == 0)


def test_zero_quants_and_mins_give_zero():
    blk = pack_block(0x3C00, 0x3C00, list(range(1, 9)), [0] * 8, [0] * 256)
    W = np.tile(blk, (2, 1))
    x = synth.activation(256, 1, 2)
    y, _ = oracle.matvec(W, oracle.quantize_q8_0(x), 2, 256)
    assert np.all(y == 0)


def test_dmin_zero_is_scaled_int8_dot():
    rng = np.random.default_rng(3)
    sc = rng.integers(0, 64, 8)
    q = rng.integers(0, 16, 256)
    blk = pack_block(0x3C00, 0x0000, sc, rng.integers(0, 64, 8), q)  # d = 1, dmin = 0
    x = synth.activation(256, 1, 3)
    xq = oracle.quantize_q8_0(x)
    y, _ = oracle.matvec(blk.reshape(1, 144), xq, 1, 256)
    dq, qi = q8_fields(xq, 256)
    expect = sum(float(dq[0, j]) * int(sc[j]) * int(np.dot(q[32 * j:32 * j + 32], qi[0, j])) for j in range(8))
    assert abs(y[0, 0] - expect) <= 1e-12 * abs(expect) + 1e-300


def test_one_hot_rows_select_activation_values():
    # row r has a single non-zero quant (value 1) at element e_r, sc = 1, m = 0, d = 1:
    # y[r] is exactly the dequantized activation value at e_r
    K = 512
    es = [0, 31, 32, 255, 256, 300, 511]
    rows = []
    for e in es:
        blocks = []
        for b in range(K // 256):
            q = np.zeros(256, np.int64)
            if e // 256 == b:
                q[e % 256] = 1
            blocks.append(pack_block(0x3C00, 0x3C00, [1] * 8, [0] * 8, q))
        rows.append(np.concatenate(blocks))
    W = np.stack(rows)
    x = synth.activation(K, 1, 4)
    xq = oracle.quantize_q8_0(x)
    y, _ = oracle.matvec(W, xq, len(es), K)
    xd = dequant_q8(xq, K)[0]
    assert np.array_equal(y[0], xd[es])


def test_min_term_sign():
    # q = 0 everywhere, sc arbitrary, m = 1, dmin = 1: every weight is -1, so y = -sum(x_hat)
    blk = pack_block(0x3C00, 0x3C00, [5] * 8, [1] * 8, [0] * 256)
    x = synth.activation(256, 1, 5)
    xq = oracle.quantize_q8_0(x)
    y, _ = oracle.matvec(blk.reshape(1, 144), xq, 1, 256)
    assert abs(y[0, 0] + dequant_q8(xq, 256)[0].sum()) <= 1e-12 * np.abs(dequant_q8(xq, 256)).sum()
