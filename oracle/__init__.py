"""CPU oracle for the q4_K x q8_0 decode matvec -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from it.  The arithmetic lives in ``mq_oracle.c``
(plain C, binary64 accumulation); this module is argument marshalling over
ctypes with numpy arrays.

Formats (a reading of the pages, which name q4_K/q8_0 but do not print them):
q4_K super-block of 256 weights in 144 bytes, q8_0 block of 32 values in 34
bytes; see ``mq_oracle.c`` for the byte layout.

Pinned by tests/test_oracle_*.py.  Nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np

from . import build as _build

QK_K = 256
Q4K_BYTES = 144
QK8 = 32
Q8_BYTES = 34

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        u8p = ctypes.POINTER(ctypes.c_uint8)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64p = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.mqo_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.mqo_f16_to_f32.restype = ctypes.c_float
        lib.mqo_f32_to_f16.argtypes = [ctypes.c_float]
        lib.mqo_f32_to_f16.restype = ctypes.c_uint16
        lib.mqo_quantize_q8_0.argtypes = [f32p, i64, u8p]
        lib.mqo_unpack_q4K.argtypes = [u8p, f64p, f64p, i32p, i32p, i32p]
        lib.mqo_dequant_q4K_row.argtypes = [u8p, i64, f64p]
        lib.mqo_dequant_q8_0.argtypes = [u8p, i64, f64p]
        lib.mqo_block_sums.argtypes = [u8p, u8p, i64, i64, i32p, i32p]
        lib.mqo_matvec.argtypes = [u8p, u8p, i64, i64, i64, f64p, f64p]
        lib.mqo_matvec_rows.argtypes = [u8p, u8p, i64, i64, i64p, i64, f64p, f64p]
        lib.mqo_silu.argtypes = [ctypes.c_double]
        lib.mqo_silu.restype = ctypes.c_double
        lib.mqo_silu_mul.argtypes = [f64p, f64p, i64, f64p]
        lib.mqo_ffn.argtypes = [u8p, u8p, f32p, i64, i64, i64, u8p, f64p, f64p, f32p, u8p, f64p]
        lib.mqo_dequant_w_row.argtypes = [ctypes.c_int, u8p, i64, f64p]
        lib.mqo_matvec_w.argtypes = [ctypes.c_int, u8p, u8p, i64, i64, i64, i64p, i64, f64p, f64p]
        lib.mqo_dequant_w_row.restype = None
        u16p = ctypes.POINTER(ctypes.c_uint16)
        lib.mqo_f64_to_f16.argtypes = [ctypes.c_double]
        lib.mqo_f64_to_f16.restype = ctypes.c_uint16
        lib.mqo_f64_to_f16_array.argtypes = [f64p, i64, u16p]
        lib.mqo_f64_to_f16_array.restype = None
        lib.mqo_dequant_q4K_f16_row.argtypes = [u8p, i64, f64p, u16p]
        lib.mqo_dequant_q4K_f16_row.restype = None
        lib.mqo_gemm_f16.argtypes = [u16p, u16p, i64, i64p, i64, i64p, i64, f64p, f64p]
        lib.mqo_gemm_f16.restype = None
        lib.mqo_matvec_w.restype = None
        for name in ("mqo_quantize_q8_0", "mqo_unpack_q4K", "mqo_dequant_q4K_row", "mqo_dequant_q8_0",
                     "mqo_block_sums", "mqo_matvec", "mqo_matvec_rows", "mqo_silu_mul", "mqo_ffn"):
            getattr(lib, name).restype = None
        _lib = lib
    return _lib


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


def f16_to_f32(bits: int) -> float:
    return float(_load().mqo_f16_to_f32(int(bits)))


def f32_to_f16(x: float) -> int:
    return int(_load().mqo_f32_to_f16(float(np.float32(x))))


def q4K_row_bytes(K: int) -> int:
    return K // QK_K * Q4K_BYTES


def q8_0_bytes(K: int) -> int:
    return K // QK8 * Q8_BYTES


def quantize_q8_0(x: np.ndarray) -> np.ndarray:
    """fp32 [ncols, K] (or [K]) -> uint8 [ncols, K/32*34] q8_0 blocks."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    x2 = x.reshape(-1, x.shape[-1])
    K = x2.shape[1]
    if K % QK8:
        raise ValueError("K must be a multiple of 32")
    out = np.empty((x2.shape[0], q8_0_bytes(K)), dtype=np.uint8)
    lib = _load()
    for c in range(x2.shape[0]):
        row = np.ascontiguousarray(x2[c])
        o = out[c]
        lib.mqo_quantize_q8_0(_p(row, ctypes.c_float), K, _p(o, ctypes.c_uint8))
    return out if x.ndim > 1 else out[0]


def unpack_q4K(block: np.ndarray) -> Tuple[float, float, np.ndarray, np.ndarray, np.ndarray]:
    """One 144-byte super-block -> (d, dmin, sc[8], m[8], q[256])."""
    b = _u8(block)
    if b.size != Q4K_BYTES:
        raise ValueError("a q4_K super-block is 144 bytes")
    d = ctypes.c_double()
    dm = ctypes.c_double()
    sc = np.zeros(8, np.int32)
    m = np.zeros(8, np.int32)
    q = np.zeros(256, np.int32)
    _load().mqo_unpack_q4K(_p(b, ctypes.c_uint8), ctypes.byref(d), ctypes.byref(dm),
                           _p(sc, ctypes.c_int32), _p(m, ctypes.c_int32), _p(q, ctypes.c_int32))
    return d.value, dm.value, sc, m, q


def dequant_q4K(W: np.ndarray, K: int) -> np.ndarray:
    """uint8 [rows, K/256*144] -> float64 [rows, K]."""
    W = _u8(W).reshape(-1, q4K_row_bytes(K))
    out = np.empty((W.shape[0], K), dtype=np.float64)
    lib = _load()
    for r in range(W.shape[0]):
        row = np.ascontiguousarray(W[r])
        o = out[r]
        lib.mqo_dequant_q4K_row(_p(row, ctypes.c_uint8), K, _p(o, ctypes.c_double))
    return out


def dequant_q8_0(xq: np.ndarray, K: int) -> np.ndarray:
    xq = _u8(xq).reshape(-1, q8_0_bytes(K))
    out = np.empty((xq.shape[0], K), dtype=np.float64)
    lib = _load()
    for c in range(xq.shape[0]):
        row = np.ascontiguousarray(xq[c])
        o = out[c]
        lib.mqo_dequant_q8_0(_p(row, ctypes.c_uint8), K, _p(o, ctypes.c_double))
    return out


def block_sums(W: np.ndarray, xq: np.ndarray, rows: int, K: int) -> Tuple[np.ndarray, np.ndarray]:
    """Per-32-block int32 sums: sumi [ncols, rows, K/32], sumq [ncols, K/32]."""
    W = _u8(W)
    xq = _u8(xq).reshape(-1, q8_0_bytes(K))
    nc = xq.shape[0]
    nq = K // QK8
    sumi = np.empty((nc, rows, nq), np.int32)
    sumq = np.empty((nc, nq), np.int32)
    lib = _load()
    for c in range(nc):
        col = np.ascontiguousarray(xq[c])
        si = sumi[c]
        sq = sumq[c]
        lib.mqo_block_sums(_p(W, ctypes.c_uint8), _p(col, ctypes.c_uint8), rows, K,
                           _p(si, ctypes.c_int32), _p(sq, ctypes.c_int32))
    return sumi, sumq


def matvec(W: np.ndarray, xq: np.ndarray, rows: int, K: int,
           row_ids: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """y, T as float64 [ncols, rows] (or [ncols, len(row_ids)]).

    T[c, r] is the sum of the magnitudes of the per-block products, the
    scale of the float tolerance |y - y_ref| <= 1e-3 * T + 1e-5.
    """
    W = _u8(W)
    xq = _u8(xq).reshape(-1, q8_0_bytes(K))
    nc = xq.shape[0]
    lib = _load()
    if row_ids is None:
        y = np.empty((nc, rows), np.float64)
        T = np.empty((nc, rows), np.float64)
        lib.mqo_matvec(_p(W, ctypes.c_uint8), _p(xq, ctypes.c_uint8), rows, K, nc,
                       _p(y, ctypes.c_double), _p(T, ctypes.c_double))
    else:
        ids = np.ascontiguousarray(row_ids, dtype=np.int64)
        if ids.size and (ids.min() < 0 or ids.max() >= rows):
            raise IndexError("row id out of range")
        y = np.empty((nc, ids.size), np.float64)
        T = np.empty((nc, ids.size), np.float64)
        lib.mqo_matvec_rows(_p(W, ctypes.c_uint8), _p(xq, ctypes.c_uint8), K, nc,
                            _p(ids, ctypes.c_int64), ids.size, _p(y, ctypes.c_double), _p(T, ctypes.c_double))
    return y, T


def silu(g: float) -> float:
    return float(_load().mqo_silu(float(g)))


def silu_mul(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    g = np.ascontiguousarray(g, dtype=np.float64)
    u = np.ascontiguousarray(u, dtype=np.float64)
    if g.shape != u.shape:
        raise ValueError("g and u must have the same shape")
    h = np.empty_like(g)
    _load().mqo_silu_mul(_p(g, ctypes.c_double), _p(u, ctypes.c_double), g.size, _p(h, ctypes.c_double))
    return h


def ffn(W_gu: np.ndarray, W_down: np.ndarray, x: np.ndarray, H: int, I: int) -> Tuple[np.ndarray, np.ndarray]:
    """Whole FFN chain: (y float64 [ncols, H], hq uint8 [ncols, I/32*34])."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, H)
    nc = x.shape[0]
    xq = np.empty(q8_0_bytes(H), np.uint8)
    gu = np.empty(2 * I, np.float64)
    h = np.empty(I, np.float64)
    hf = np.empty(I, np.float32)
    hq = np.empty((nc, q8_0_bytes(I)), np.uint8)
    y = np.empty((nc, H), np.float64)
    _load().mqo_ffn(_p(_u8(W_gu), ctypes.c_uint8), _p(_u8(W_down), ctypes.c_uint8), _p(x, ctypes.c_float),
                    H, I, nc, _p(xq, ctypes.c_uint8), _p(gu, ctypes.c_double), _p(h, ctypes.c_double),
                    _p(hf, ctypes.c_float), _p(hq, ctypes.c_uint8), _p(y, ctypes.c_double))
    return y, hq


def within_tolerance(y: np.ndarray, y_ref: np.ndarray, T: np.ndarray) -> np.ndarray:
    """|y - y_ref| <= 1e-3 * T + 1e-5, elementwise."""
    return np.abs(np.asarray(y, np.float64) - y_ref) <= 1e-3 * T + 1e-5


# ---- 32-weight block types: q4_0 (18 bytes) and q8_0 (34 bytes) weights ------------------------------------

W_BLOCK_BYTES = {"q4_0": 18, "q8_0": 34}


def w_row_bytes(wtype: str, K: int) -> int:
    return K // QK8 * W_BLOCK_BYTES[wtype]


def dequant_w_row(wtype: str, row: np.ndarray, K: int) -> np.ndarray:
    """One row of K weights of a 32-weight block type -> binary64."""
    row = _u8(row).reshape(-1)
    if row.size != w_row_bytes(wtype, K):
        raise ValueError("row size does not match K")
    out = np.empty(K, np.float64)
    _load().mqo_dequant_w_row(W_BLOCK_BYTES[wtype], _p(row, ctypes.c_uint8), K, _p(out, ctypes.c_double))
    return out


def matvec_w(wtype: str, W: np.ndarray, xq: np.ndarray, rows: int, K: int,
             row_ids: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """y, T [ncols, rows or len(row_ids)] for q4_0 / q8_0 weights and q8_0 activations, fp64."""
    W = _u8(W).reshape(-1)
    xq2 = _u8(xq).reshape(-1, q8_0_bytes(K))
    ncols = xq2.shape[0]
    if W.size != rows * w_row_bytes(wtype, K):
        raise ValueError("W size does not match rows x K")
    ids = None if row_ids is None else np.ascontiguousarray(row_ids, dtype=np.int64)
    n = rows if ids is None else ids.size
    y = np.empty((ncols, n), np.float64)
    T = np.empty((ncols, n), np.float64)
    _load().mqo_matvec_w(W_BLOCK_BYTES[wtype], _p(W, ctypes.c_uint8), _p(np.ascontiguousarray(xq2), ctypes.c_uint8),
                         rows, K, ncols, None if ids is None else _p(ids, ctypes.c_int64), n,
                         _p(y, ctypes.c_double), _p(T, ctypes.c_double))
    return y, T


# ---- prefill: the f16 weight cache and the half-precision GEMM ---------------------------------------------

def f64_to_f16(x) -> np.ndarray:
    """binary64 values -> binary16 bit patterns (uint16), round to nearest, ties to even."""
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(a.shape, np.uint16)
    _load().mqo_f64_to_f16_array(_p(a.reshape(-1), ctypes.c_double), a.size,
                                 _p(out.reshape(-1), ctypes.c_uint16))
    return out


def dequant_q4K_f16(W: np.ndarray, K: int) -> np.ndarray:
    """uint8 q4_K [rows, K/256*144] -> uint16 binary16 patterns [rows, K] (each weight rounded once)."""
    W = _u8(W).reshape(-1, q4K_row_bytes(K))
    out = np.empty((W.shape[0], K), np.uint16)
    scratch = np.empty(K, np.float64)
    lib = _load()
    for r in range(W.shape[0]):
        row = np.ascontiguousarray(W[r])
        o = out[r]
        lib.mqo_dequant_q4K_f16_row(_p(row, ctypes.c_uint8), K, _p(scratch, ctypes.c_double),
                                    _p(o, ctypes.c_uint16))
    return out


def f32_to_f16_array(x) -> np.ndarray:
    """fp32 values -> binary16 bit patterns (uint16), round to nearest, ties to even."""
    return f64_to_f16(np.asarray(x, np.float32).astype(np.float64))


def gemm_f16(W16: np.ndarray, X16: np.ndarray, K: int, row_ids=None, tok_ids=None) -> Tuple[np.ndarray, np.ndarray]:
    """Y [len(tok_ids), len(row_ids)] = X16 . W16^T over the chosen tokens and rows, binary64 sums of the
    exact binary16 products; and T, the sums of the products' magnitudes.  W16 uint16 [R, K], X16 uint16 [T, K]."""
    W16 = np.ascontiguousarray(W16, dtype=np.uint16).reshape(-1, K)
    X16 = np.ascontiguousarray(X16, dtype=np.uint16).reshape(-1, K)
    rows = np.arange(W16.shape[0], dtype=np.int64) if row_ids is None else np.ascontiguousarray(row_ids, np.int64)
    toks = np.arange(X16.shape[0], dtype=np.int64) if tok_ids is None else np.ascontiguousarray(tok_ids, np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= W16.shape[0]):
        raise IndexError("row id out of range")
    if toks.size and (toks.min() < 0 or toks.max() >= X16.shape[0]):
        raise IndexError("token id out of range")
    y = np.empty((toks.size, rows.size), np.float64)
    T = np.empty((toks.size, rows.size), np.float64)
    _load().mqo_gemm_f16(_p(W16, ctypes.c_uint16), _p(X16, ctypes.c_uint16), K, _p(rows, ctypes.c_int64),
                         rows.size, _p(toks, ctypes.c_int64), toks.size, _p(y, ctypes.c_double),
                         _p(T, ctypes.c_double))
    return y, T
