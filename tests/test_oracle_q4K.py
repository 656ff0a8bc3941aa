"""Pins for the oracle's q4_K super-block unpack.

The pages name q4_K ("07 . R3", section 1) without printing it; the layout is
the GGUF-compatible reading.  Pins: (1) the bit structure -- every one of the
96 scale bits and 1024 quant bits moves exactly one logical field by one
power of two, each (field, bit) exactly once; (2) single-bit placements stated
in the reading; (3) an exhaustive round trip through an independent packer;
(4) the closed form for all-equal fields.
"""
import numpy as np
import pytest

import oracle
from tests.q4k_layout import pack_block, unpack_fields


def _fields(block):
    d, dmin, sc, m, q = oracle.unpack_q4K(block)
    return d, dmin, np.array(sc), np.array(m), np.array(q)


def _random_block(rng):
    b = rng.integers(0, 256, 144, dtype=np.uint8)
    b[0:2] = np.array([np.float16(1.5e-3)]).view(np.uint8)
    b[2:4] = np.array([np.float16(7e-4)]).view(np.uint8)
    return b


def test_scale_bits_form_a_bijection():
    rng = np.random.default_rng(1)
    base = _random_block(rng)
    _, _, sc0, m0, q0 = _fields(base)
    seen = set()
    for byte in range(4, 16):
        for bit in range(8):
            b = base.copy()
            b[byte] ^= np.uint8(1 << bit)
            _, _, sc, m, q = _fields(b)
            assert np.array_equal(q, q0)
            dsc = np.nonzero(sc != sc0)[0]
            dm = np.nonzero(m != m0)[0]
            assert len(dsc) + len(dm) == 1, (byte, bit)
            if len(dsc):
                j, delta, kind = dsc[0], abs(int(sc[dsc[0]]) - int(sc0[dsc[0]])), "sc"
            else:
                j, delta, kind = dm[0], abs(int(m[dm[0]]) - int(m0[dm[0]])), "m"
            k = int(delta).bit_length() - 1
            assert delta == 1 << k and 0 <= k < 6
            seen.add((kind, int(j), k))
    assert len(seen) == 96


def test_quant_bits_form_a_bijection():
    rng = np.random.default_rng(2)
    base = _random_block(rng)
    _, _, sc0, m0, q0 = _fields(base)
    seen = set()
    for byte in range(16, 144):
        for bit in range(8):
            b = base.copy()
            b[byte] ^= np.uint8(1 << bit)
            _, _, sc, m, q = _fields(b)
            assert np.array_equal(sc, sc0) and np.array_equal(m, m0)
            diff = np.nonzero(q != q0)[0]
            assert len(diff) == 1
            delta = abs(int(q[diff[0]]) - int(q0[diff[0]]))
            k = delta.bit_length() - 1
            assert delta == 1 << k and k < 4
            seen.add((int(diff[0]), k))
    assert len(seen) == 1024


def test_quant_nibble_placement():
    base = np.zeros(144, np.uint8)
    for c in range(4):
        for i in (0, 5, 31):
            b = base.copy()
            b[16 + 32 * c + i] = 0x01              # low nibble: element i of sub-block 2c
            q = _fields(b)[4]
            assert np.nonzero(q)[0].tolist() == [64 * c + i]
            b[16 + 32 * c + i] = 0x10              # high nibble: element i of sub-block 2c+1
            q = _fields(b)[4]
            assert np.nonzero(q)[0].tolist() == [64 * c + 32 + i]


def test_scale_byte_placement():
    z = np.zeros(144, np.uint8)
    for j in range(4):
        b = z.copy(); b[4 + j] = 0x3F
        _, _, sc, m, _ = _fields(b)
        assert sc.tolist() == [63 if t == j else 0 for t in range(8)] and not m.any()
        b = z.copy(); b[8 + j] = 0x3F
        _, _, sc, m, _ = _fields(b)
        assert m.tolist() == [63 if t == j else 0 for t in range(8)] and not sc.any()
        # top two bits of scale byte j are bits 4-5 of sc_{j+4}
        b = z.copy(); b[4 + j] = 0xC0
        _, _, sc, m, _ = _fields(b)
        assert sc.tolist() == [48 if t == j + 4 else 0 for t in range(8)] and not m.any()
        # top two bits of scale byte j+4 are bits 4-5 of m_{j+4}
        b = z.copy(); b[8 + j] = 0xC0
        _, _, sc, m, _ = _fields(b)
        assert m.tolist() == [48 if t == j + 4 else 0 for t in range(8)] and not sc.any()
        # scale byte j+8: low nibble -> sc_{j+4} bits 0-3, high nibble -> m_{j+4} bits 0-3
        b = z.copy(); b[12 + j] = 0x5A
        _, _, sc, m, _ = _fields(b)
        assert sc.tolist() == [0xA if t == j + 4 else 0 for t in range(8)]
        assert m.tolist() == [0x5 if t == j + 4 else 0 for t in range(8)]


def test_d_dmin_little_endian_binary16():
    rng = np.random.default_rng(3)
    for _ in range(100):
        b = rng.integers(0, 256, 144, dtype=np.uint8)
        b[1] &= 0x7B  # keep finite
        b[3] &= 0x7B
        d, dmin, *_ = _fields(b)
        assert d == float(b[0:2].view(np.float16)[0])
        assert dmin == float(b[2:4].view(np.float16)[0])


def test_exhaustive_scale_roundtrip_every_position():
    rng = np.random.default_rng(4)
    q = rng.integers(0, 16, 256)
    for j in range(8):
        for s in range(64):
            for mv in range(0, 64, 1 if j in (0, 4, 7) else 9):
                sc = rng.integers(0, 64, 8)
                m = rng.integers(0, 64, 8)
                sc[j] = s
                m[j] = mv
                blk = pack_block(0x3C00, 0x3800, sc, m, q)
                _, _, sc2, m2, q2 = _fields(blk)
                assert np.array_equal(sc2, sc) and np.array_equal(m2, m) and np.array_equal(q2, q)


def test_matches_independent_numpy_unpack_random():
    rng = np.random.default_rng(5)
    blocks = rng.integers(0, 256, (300, 144), dtype=np.uint8)
    blocks[:, 1] &= 0x7B
    blocks[:, 3] &= 0x7B
    d, dmin, sc, m, q = unpack_fields(blocks)
    for t in range(300):
        d2, dmin2, sc2, m2, q2 = _fields(blocks[t])
        assert d2 == d[t] and dmin2 == dmin[t]
        assert np.array_equal(sc2, sc[t]) and np.array_equal(m2, m[t]) and np.array_equal(q2, q[t])


@pytest.mark.parametrize("qv,s,mv", [(0, 0, 0), (15, 63, 63), (7, 1, 0), (1, 63, 5), (9, 17, 44)])
@pytest.mark.parametrize("d_bits,dmin_bits", [(0x3C00, 0x3800), (0x1234, 0x0007), (0x0001, 0x03FF)])
def test_closed_form_all_equal(qv, s, mv, d_bits, dmin_bits):
    # every element dequantizes to d*s*q - dmin*m, exactly: d*s*q has at most
    # 11+6+4 significant bits and dmin*m at most 11+6, so binary64 is exact
    blk = pack_block(d_bits, dmin_bits, [s] * 8, [mv] * 8, [qv] * 256)
    w = oracle.dequant_q4K(blk.reshape(1, 144), 256)[0]
    d = float(np.uint16(d_bits).view(np.float16))
    dmin = float(np.uint16(dmin_bits).view(np.float16))
    expect = d * s * qv - dmin * mv
    assert np.all(w == expect)
