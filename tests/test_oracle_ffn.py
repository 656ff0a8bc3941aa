"""Pins for the oracle's SiLU and FFN chain.

The FFN ("04 . 8o", sections 1 and 3.1) multiplies by ffn_gu, gate rows first
then up rows, applies SwiGLU and then down.  Checked against scipy's logistic
function and an independent numpy composition (numpy unpack + matmul).
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from quantized_decode_matvec_gb300 import synth
from tests.q4k_layout import dequant_q8, dequant_rows, pack_block


def test_silu_special_values():
    assert oracle.silu(0.0) == 0.0
    assert abs(oracle.silu(40.0) - 40.0) < 1e-12
    s = oracle.silu(-40.0)
    assert s < 0 and abs(s) < 1e-15
    for g in np.linspace(-30, 30, 121):
        assert abs(oracle.silu(g) - g * expit(g)) <= 1e-15 * max(1.0, abs(g))


def test_silu_mul_matches_scipy():
    rng = np.random.default_rng(0)
    g = rng.standard_normal(1000) * 5
    u = rng.standard_normal(1000)
    h = oracle.silu_mul(g, u)
    assert np.allclose(h, g * expit(g) * u, rtol=1e-14, atol=0)


def _independent_ffn(W_gu, W_down, x, H, I):
    xq = oracle.quantize_q8_0(x)
    gu = dequant_rows(W_gu, H) @ dequant_q8(xq, H)[0]
    g, u = gu[:I], gu[I:]
    h = (g * expit(g) * u).astype(np.float32)
    hq = oracle.quantize_q8_0(h.reshape(1, -1))
    y = dequant_rows(W_down, I) @ dequant_q8(hq, I)[0]
    return y, hq[0]


def test_ffn_chain_matches_independent_composition():
    H, I = 512, 256
    W_gu = synth.q4K_matrix(2 * I, H, 9, synth.TAG_GU)
    W_down = synth.q4K_matrix(H, I, 9, synth.TAG_DOWN)
    x = synth.activation(H, 2, 9)
    y, hq = oracle.ffn(W_gu, W_down, x, H, I)
    for c in range(2):
        y_ref, hq_ref = _independent_ffn(W_gu, W_down, x[c:c + 1], H, I)
        # h is re-quantized: a last-ulp difference in h could flip a q8 code, so
        # compare the codes exactly where they agree and y loosely
        same = np.mean(hq[c] == hq_ref)
        assert same > 0.99
        _, T = oracle.matvec(W_down, hq[c:c + 1], H, I)
        assert np.all(np.abs(y[c] - y_ref) <= 1e-3 * T[0] + 1e-5)


def test_ffn_gate_rows_come_first():
    # gate half of ffn_gu zero (sc = m = 0) -> g = 0 -> SiLU(0) = 0 -> h = 0, whatever up is;
    # a swapped gate/up order would give h = SiLU(u) * 0 = 0 too, so also check the converse:
    # up half zero -> h = 0; gate half zero with up non-zero -> h = 0; both non-zero -> h != 0.
    H, I = 256, 256
    zero_row = pack_block(0x3C00, 0x3C00, [0] * 8, [0] * 8, [3] * 256)
    rng = np.random.default_rng(1)
    live = synth.q4K_matrix(I, H, 2, synth.TAG_GU)
    W_down = synth.q4K_matrix(H, I, 2, synth.TAG_DOWN)
    x = synth.activation(H, 1, 2)
    zeros = np.tile(zero_row, (I, 1))
    # gate = live, up = ones-like constant rows: weights all d*sc*q with sc = 1
    up_const = np.tile(pack_block(0x3C00, 0x3C00, [1] * 8, [0] * 8, [1] * 256), (I, 1))
    y_a, hq_a = oracle.ffn(np.concatenate([live, up_const]), W_down, x, H, I)
    y_b, hq_b = oracle.ffn(np.concatenate([up_const, live]), W_down, x, H, I)
    # with gate = live, h = SiLU(live.x) * sum(x_hat); with gate = const, h = SiLU(sum(x_hat)) * live.x
    xq = oracle.quantize_q8_0(x)
    s = dequant_q8(xq, H)[0].sum()
    g_live = dequant_rows(live, H) @ dequant_q8(xq, H)[0]
    h_a = (g_live * expit(g_live) * s).astype(np.float32)
    h_b = (s * expit(s) * g_live).astype(np.float32)
    assert np.mean(hq_a[0] == oracle.quantize_q8_0(h_a.reshape(1, -1))[0]) > 0.99
    assert np.mean(hq_b[0] == oracle.quantize_q8_0(h_b.reshape(1, -1))[0]) > 0.99
    y0, hq0 = oracle.ffn(np.concatenate([zeros, live]), W_down, x, H, I)
    assert np.all(y0 == 0) and np.all(hq0 == 0)
