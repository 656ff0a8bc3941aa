"""Test-side pack/unpack of the q4_K and q8_0 byte layouts, vectorized numpy.

Written from the layout's description (the GGUF-compatible reading), not from
the oracle's code, so that the oracle's loop-based C unpacker can be checked
against an independent implementation.  Used only by tests.

q4_K super-block (144 B): [0:2] d f16, [2:4] dmin f16, [4:16] twelve scale
bytes, [16:144] 128 quant bytes.  Scale bytes: bytes 0-3 carry sc0..sc3 in
their low 6 bits, bytes 4-7 carry m0..m3 the same way; the top two bits of
bytes 0-3 are bits 4-5 of sc4..sc7, the top two bits of bytes 4-7 are bits
4-5 of m4..m7; bytes 8-11 carry bits 0-3 of sc4..sc7 (low nibble) and of
m4..m7 (high nibble).  Quant bytes: 4 chunks of 32; byte i of chunk c holds
element i of sub-block 2c (low nibble) and of sub-block 2c+1 (high nibble).
"""
import numpy as np


def unpack_fields(blocks: np.ndarray):
    """uint8 [..., 144] -> d f64, dmin f64, sc [..., 8], m [..., 8], q [..., 256]."""
    b = np.asarray(blocks, dtype=np.uint8)
    d = b[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    dmin = b[..., 2:4].copy().view(np.float16)[..., 0].astype(np.float64)
    s = b[..., 4:16].astype(np.int64)
    lo6 = s[..., 0:4] & 63
    mlo6 = s[..., 4:8] & 63
    top_sc = s[..., 0:4] >> 6
    top_m = s[..., 4:8] >> 6
    sc_hi = (s[..., 8:12] & 15) | (top_sc << 4)
    m_hi = (s[..., 8:12] >> 4) | (top_m << 4)
    sc = np.concatenate([lo6, sc_hi], axis=-1)
    m = np.concatenate([mlo6, m_hi], axis=-1)
    qs = b[..., 16:144].astype(np.int64).reshape(b.shape[:-1] + (4, 32))
    lo = qs & 15                      # sub-block 2c
    hi = qs >> 4                      # sub-block 2c+1
    q = np.stack([lo, hi], axis=-2).reshape(b.shape[:-1] + (256,))
    return d, dmin, sc, m, q


def pack_block(d_bits: int, dmin_bits: int, sc, m, q) -> np.ndarray:
    """Logical fields -> one 144-byte super-block."""
    sc = np.asarray(sc, np.int64)
    m = np.asarray(m, np.int64)
    q = np.asarray(q, np.int64).reshape(8, 32)
    assert sc.shape == (8,) and m.shape == (8,)
    assert (sc >= 0).all() and (sc < 64).all() and (m >= 0).all() and (m < 64).all()
    assert (q >= 0).all() and (q < 16).all()
    out = np.zeros(144, np.uint8)
    out[0] = d_bits & 0xFF
    out[1] = d_bits >> 8
    out[2] = dmin_bits & 0xFF
    out[3] = dmin_bits >> 8
    s = np.zeros(12, np.int64)
    s[0:4] = sc[0:4] | ((sc[4:8] >> 4) << 6)
    s[4:8] = m[0:4] | ((m[4:8] >> 4) << 6)
    s[8:12] = (sc[4:8] & 15) | ((m[4:8] & 15) << 4)
    out[4:16] = s.astype(np.uint8)
    chunks = q.reshape(4, 2, 32)
    out[16:144] = (chunks[:, 0, :] | (chunks[:, 1, :] << 4)).reshape(128).astype(np.uint8)
    return out


def dequant_rows(W: np.ndarray, K: int) -> np.ndarray:
    """uint8 [rows, K/256*144] -> float64 [rows, K] via unpack_fields."""
    rows = W.shape[0]
    blocks = W.reshape(rows, K // 256, 144)
    d, dmin, sc, m, q = unpack_fields(blocks)
    qv = q.reshape(rows, K // 256, 8, 32).astype(np.float64)
    w = d[..., None, None] * sc[..., None].astype(np.float64) * qv - dmin[..., None, None] * m[..., None].astype(np.float64)
    return w.reshape(rows, K)


def q8_fields(xq: np.ndarray, K: int):
    """uint8 [ncols, K/32*34] -> scales f64 [ncols, K/32], ints [ncols, K/32, 32]."""
    b = np.asarray(xq, np.uint8).reshape(-1, K // 32, 34)
    dq = b[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    qi = b[..., 2:34].copy().view(np.int8).astype(np.int64)
    return dq, qi


def dequant_q8(xq: np.ndarray, K: int) -> np.ndarray:
    dq, qi = q8_fields(xq, K)
    return (dq[..., None] * qi).reshape(dq.shape[0], K)
