"""Seeded synthetic inputs for the q4_K x q8_0 decode matvec workloads.

This module only draws random bytes and floats. It holds none of the
method's arithmetic: it never quantizes, packs, unpacks or multiplies, so
that the CPU oracle and the CUDA path can both consume its output without
sharing any code with each other.

Recipe (every tensor gets its own stream, ``PCG64(SeedSequence([seed, tag]))``):

* q4_K weight matrix [rows, K] (K a multiple of 256): ``rows * K/256``
  super-blocks of 144 bytes.  First the whole byte image is drawn uniformly
  (the raw 64-bit PCG64 outputs, ``bit_generator.random_raw``, read as
  little-endian bytes), then bytes 0-1 of every super-block are overwritten
  with the binary16 value of ``|N(0, 2e-3)|`` (the super-block scale d) and
  bytes 2-3 with binary16 ``|N(0, 1e-3)|`` (dmin), both converted by numpy's
  ``astype(float16)``.  Because the twelve scale bytes carry exactly sixteen
  6-bit fields and the 128 quant bytes exactly 256 4-bit fields, uniform
  bytes give scales/mins uniform in 0..63 and quants uniform in 0..15, which
  is the distribution the workloads specify, without packing anything here.
  Small draws of d/dmin land on binary16 subnormals (about 3 % of blocks).
* fp32 activation [ncols, K]: ``standard_normal(dtype=float32)``, then each
  entry independently with probability 1e-3 (``random() < 1e-3`` from the
  same stream) is multiplied by 20.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import numpy as np

QK_K = 256          # weights per q4_K super-block
Q4K_BLOCK_BYTES = 144
QK8_0 = 32          # values per q8_0 block
Q8_0_BLOCK_BYTES = 34

# tags that name each tensor's random stream
TAG_W = 1
TAG_X = 2
TAG_GU = 3
TAG_DOWN = 4
TAG_Q = 5
TAG_K = 6
TAG_V = 7
TAG_O = 8
TAG_A = 9      # step: input of the q/k/v projections
TAG_B = 10     # step: input of the o projection
TAG_C = 11     # step: input of the FFN
TAG_COLS = 12  # multi-column activations


def stream(seed: int, tag: int, layer: int = 0, extra: int = 0) -> np.random.Generator:
    """Independent PCG64 stream for one tensor."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, layer, extra])))


def q4K_matrix(rows: int, K: int, seed: int, tag: int = TAG_W, layer: int = 0,
               d_sigma: float = 2e-3, dmin_sigma: float = 1e-3) -> np.ndarray:
    """Random q4_K matrix as uint8 [rows, K/256*144] (row-major, rows contiguous)."""
    if K % QK_K:
        raise ValueError("K must be a multiple of 256")
    nb = K // QK_K
    rng = stream(seed, tag, layer)
    nbytes = rows * nb * Q4K_BLOCK_BYTES
    raw = rng.bit_generator.random_raw((nbytes + 7) // 8).astype("<u8", copy=False)
    img = raw.view(np.uint8)[:nbytes].reshape(rows * nb, Q4K_BLOCK_BYTES)
    d = np.abs(rng.standard_normal(rows * nb)) * d_sigma
    dmin = np.abs(rng.standard_normal(rows * nb)) * dmin_sigma
    img[:, 0:2] = d.astype(np.float16).view(np.uint8).reshape(-1, 2)
    img[:, 2:4] = dmin.astype(np.float16).view(np.uint8).reshape(-1, 2)
    return img.reshape(rows, nb * Q4K_BLOCK_BYTES)


# 32-weight block types of the pages' other models: block bytes, default scale sigma
WBLOCK = {"q4_0": (18, 2e-3), "q8_0": (34, 2e-4)}
TAG_WQ = 13  # q4_0 / q8_0 weight matrices


def wq_matrix(wtype: str, rows: int, K: int, seed: int, tag: int = TAG_WQ, layer: int = 0,
              d_sigma: float | None = None) -> np.ndarray:
    """Random q4_0 or q8_0 weight matrix as uint8 [rows, K/32*block_bytes]: uniform bytes, then
    bytes 0-1 of every block overwritten with binary16 |N(0, d_sigma)| (the block scale)."""
    if K % QK8_0:
        raise ValueError("K must be a multiple of 32")
    bb, sigma = WBLOCK[wtype]
    nb = K // QK8_0
    rng = stream(seed, tag, layer, bb)
    nbytes = rows * nb * bb
    raw = rng.bit_generator.random_raw((nbytes + 7) // 8).astype("<u8", copy=False)
    img = raw.view(np.uint8)[:nbytes].reshape(rows * nb, bb)
    d = np.abs(rng.standard_normal(rows * nb)) * (sigma if d_sigma is None else d_sigma)
    img[:, 0:2] = d.astype(np.float16).view(np.uint8).reshape(-1, 2)
    return img.reshape(rows, nb * bb)


def activation(K: int, ncols: int, seed: int, tag: int = TAG_X, layer: int = 0,
               outlier_p: float = 1e-3, outlier_scale: float = 20.0) -> np.ndarray:
    """fp32 [ncols, K] N(0,1) activation with sparse x20 outliers."""
    rng = stream(seed, tag, layer)
    x = rng.standard_normal((ncols, K), dtype=np.float32)
    mask = rng.random((ncols, K)) < outlier_p
    x[mask] *= np.float32(outlier_scale)
    return x


# --------------------------------------------------------------------------------------
# The workloads, by what they are.  Shapes are (rows, K) with K the reduction length.
# --------------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class MatvecCase:
    name: str
    rows: int
    K: int
    ncols: int
    seed: int


@dataclasses.dataclass(frozen=True)
class FfnCase:
    name: str
    H: int          # hidden (K of ffn_gu, rows of down)
    I: int          # intermediate (ffn_gu has 2I rows, down has K = I)
    ncols: int
    n_layers: int
    seed: int


@dataclasses.dataclass(frozen=True)
class StepCase:
    name: str
    n_layers: int
    H: int
    I: int
    q_rows: int
    kv_rows: int
    ncols: int
    seed: int

    @property
    def qkv_rows(self) -> int:
        return self.q_rows + 2 * self.kv_rows


# single q4_K x q8_0 matvec, 512 rows x K=1024, one column, seed 0
MATVEC_512x1024 = MatvecCase("matvec_512x1024", 512, 1024, 1, 0)
# 0.5B-class decode FFN, 24 layers, hidden 1024, intermediate 4864, seed 0
FFN_05B = FfnCase("ffn_0.5B_h1024_i4864_x24", 1024, 4864, 1, 24, 0)
# 7B-class decode FFN, one layer, hidden 3584, intermediate 18944, seed 1
FFN_7B = FfnCase("ffn_7B_h3584_i18944", 3584, 18944, 1, 1, 1)
# 7B-class whole decode step of matvecs, 28 layers, seed 2
STEP_7B = StepCase("step_7B_28L", 28, 3584, 18944, 3584, 512, 1, 2)
# multi-sequence decode on the 7B FFN weights (seed 1 weights, own column streams)
FFN_7B_NCOLS = (2, 4, 8)
# K sweep on a 4096-row matrix, one column, seed 3
KSWEEP_ROWS = 4096
KSWEEP_KS = (1024, 4096, 14336, 18944)
KSWEEP_SEED = 3


def matvec_case_inputs(case: MatvecCase) -> Tuple[np.ndarray, np.ndarray]:
    W = q4K_matrix(case.rows, case.K, case.seed, TAG_W)
    x = activation(case.K, case.ncols, case.seed, TAG_X)
    return W, x


def ffn_layer_weights(case: FfnCase, layer: int) -> Tuple[np.ndarray, np.ndarray]:
    """(W_gu [2I, H] gate rows then up rows, W_down [H, I]) for one layer."""
    W_gu = q4K_matrix(2 * case.I, case.H, case.seed, TAG_GU, layer)
    W_down = q4K_matrix(case.H, case.I, case.seed, TAG_DOWN, layer)
    return W_gu, W_down


def ffn_layer_input(case: FfnCase, layer: int, ncols: int | None = None) -> np.ndarray:
    nc = case.ncols if ncols is None else ncols
    tag = TAG_X if nc == 1 else TAG_COLS
    return activation(case.H, nc, case.seed, tag, layer)


def step_layer_weights(case: StepCase, layer: int, d_scale: float = 1.0,
                       dmin_scale: float | None = None) -> Dict[str, np.ndarray]:
    """The six q4_K projections of one layer (q, k, v, o, ffn_gu, down).

    d_scale and dmin_scale multiply the standard deviations of d and dmin
    (1.0: the workloads' |N(0, 2e-3)| and |N(0, 1e-3)|; dmin_scale defaults to
    d_scale).  A chain of layers with no normalization between them changes
    its scale by a factor per projection that is proportional to them; with
    the workloads' draws the weights' mean is d*31.5*7.5 - dmin*31.5 > 0, a
    component common to every row that grows by about K times that mean per
    projection.  A chain test takes dmin_scale = 15 * d_scale (mean about zero)
    and a small d_scale, which keeps a short chain's values of order one."""
    H, I = case.H, case.I
    kw = dict(d_sigma=2e-3 * d_scale, dmin_sigma=1e-3 * (d_scale if dmin_scale is None else dmin_scale))
    return {
        "q": q4K_matrix(case.q_rows, H, case.seed, TAG_Q, layer, **kw),
        "k": q4K_matrix(case.kv_rows, H, case.seed, TAG_K, layer, **kw),
        "v": q4K_matrix(case.kv_rows, H, case.seed, TAG_V, layer, **kw),
        "o": q4K_matrix(H, case.q_rows, case.seed, TAG_O, layer, **kw),
        "gu": q4K_matrix(2 * I, H, case.seed, TAG_GU, layer, **kw),
        "down": q4K_matrix(H, I, case.seed, TAG_DOWN, layer, **kw),
    }


def step_layer_inputs(case: StepCase, layer: int, replay: int = 0) -> Dict[str, np.ndarray]:
    """Per-layer fp32 inputs a (feeds q|k|v), b (feeds o), c (feeds the FFN).

    ``replay`` selects a fresh draw for each graph replay.
    """
    out = {}
    for name, tag in (("a", TAG_A), ("b", TAG_B), ("c", TAG_C)):
        rng_layer = layer + 1000 * replay
        K = case.H if name != "b" else case.q_rows
        out[name] = activation(K, case.ncols, case.seed, tag, rng_layer)
    return out


def ksweep_inputs(K: int) -> Tuple[np.ndarray, np.ndarray]:
    W = q4K_matrix(KSWEEP_ROWS, K, KSWEEP_SEED, TAG_W, layer=K)
    x = activation(K, 1, KSWEEP_SEED, TAG_X, layer=K)
    return W, x


def weight_bytes_step(case: StepCase) -> int:
    H, I = case.H, case.I
    per_row = lambda K: K // QK_K * Q4K_BLOCK_BYTES
    per_layer = (case.qkv_rows * per_row(H) + H * per_row(case.q_rows)
                 + 2 * I * per_row(H) + H * per_row(I))
    return per_layer * case.n_layers


def weight_bytes_ffn(case: FfnCase) -> int:
    per_row = lambda K: K // QK_K * Q4K_BLOCK_BYTES
    return (2 * case.I * per_row(case.H) + case.H * per_row(case.I)) * case.n_layers


__all__ = [n for n in dir() if not n.startswith("_")]
