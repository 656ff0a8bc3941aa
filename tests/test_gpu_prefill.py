"""Prefill on the GPU ("07 . R3 -- Small-model per-token overhead", section 1: a
half-precision tensor-core GEMM over a resident f16 copy of the weights).

Bars: the f16 weight cache and the f16 activations are bit-exact with the
oracle (each value rounded once, to nearest-even); the GEMM's fp32 outputs are
within |y - y_ref| <= 1e-3 * T + 1e-5 of the oracle's binary64 sums, T the
sum of the products' magnitudes, and in fact within the fp32 accumulation
bound 2e-5 * T + 1e-6 (checked too: a misplaced tile or K-step would be far
outside either).
"""
import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _u16(t):
    import torch
    torch.cuda.synchronize()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("rows,K,d_sigma", [(7, 256, 2e-3), (300, 3584, 2e-3), (64, 18944, 2e-3),
                                            (40, 512, 100.0)])
def test_dequant_f16_bit_exact(cuda_ready, rows, K, d_sigma):
    # d_sigma 100: weights beyond the f16 range round to infinity on both sides
    mq = cuda_ready
    W = synth.q4K_matrix(rows, K, seed=rows + K, d_sigma=d_sigma, dmin_sigma=d_sigma / 2)
    got = _u16(mq.dequant_q4K_f16(_dev(W), rows, K))
    assert np.array_equal(got, oracle.dequant_q4K_f16(W, K))


def test_convert_f32_f16_bit_exact(cuda_ready):
    mq = cuda_ready
    rng = np.random.default_rng(70)
    x = np.concatenate([
        synth.activation(4096, 3, seed=71).reshape(-1),
        (rng.standard_normal(50000) * np.exp2(rng.uniform(-30, 17, 50000))).astype(np.float32),
        # binary16 midpoints (exact in fp32 for normal f16 values) and the overflow edge
        ((np.arange(1, 2000, dtype=np.uint16).view(np.float16).astype(np.float32)
          + np.arange(2, 2001, dtype=np.uint16).view(np.float16).astype(np.float32)) / 2),
        np.array([65504.0, 65519.996, 65520.0, -65520.0, 0.0, -0.0, 1e-30], np.float32),
    ]).astype(np.float32)
    got = _u16(mq.convert_f32_f16(_dev(x)))
    assert np.array_equal(got, oracle.f32_to_f16_array(x))


def _gemm_case(R, K, T, seed):
    """f16 operands: the cache of a random q4_K matrix when K is a multiple of 256, else
    binary16 roundings of N(0, 0.05^2) weights; activations as the workloads draw them."""
    if K % 256 == 0:
        W16 = oracle.dequant_q4K_f16(synth.q4K_matrix(R, K, seed=seed), K)
    else:
        W16 = oracle.f64_to_f16(np.random.default_rng(seed).standard_normal((R, K)) * 0.05)
    x = synth.activation(K, T, seed=seed + 1)
    return W16, oracle.f32_to_f16_array(x)


def _check(y, W16, X16, K, rows=None, toks=None):
    y_ref, Tm = oracle.gemm_f16(W16, X16, K, row_ids=rows, tok_ids=toks)
    yg = y if rows is None else y[np.ix_(toks, rows)]
    err = np.abs(yg.astype(np.float64) - y_ref)
    assert oracle.within_tolerance(yg, y_ref, Tm).all()
    assert (err <= 2e-5 * Tm + 1e-6).all(), float((err / (Tm + 1e-30)).max())


# one tile; several K-steps; both accumulators of a CTA; ragged rows and tokens; one row and token
GEMM_SHAPES = [(128, 64, 256), (128, 512, 256), (256, 256, 1024), (200, 192, 300), (1, 64, 1), (384, 1024, 700)]


@pytest.mark.parametrize("R,K,T", GEMM_SHAPES)
def test_gemm_f16_small(cuda_ready, R, K, T):
    import torch
    mq = cuda_ready
    W16, X16 = _gemm_case(R, K, T, seed=R * 3 + K + T)
    Y = torch.full((T, R), float("nan"), dtype=torch.float32, device="cuda")
    mq.gemm_f16(_dev(W16.view(np.float16)), _dev(X16.view(np.float16)), out=Y)
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    _check(Y.cpu().numpy(), W16, X16, K)


def test_gemm_f16_many_tiles_per_cta(cuda_ready):
    # more tiles than CTAs: every CTA walks several tiles and reuses both accumulators
    import torch
    mq = cuda_ready
    R, K, T = 4608, 256, 2048
    W16, X16 = _gemm_case(R, K, T, seed=81)
    Y = mq.gemm_f16(_dev(W16.view(np.float16)), _dev(X16.view(np.float16)))
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    rng = np.random.default_rng(82)
    rows = np.unique(np.concatenate([rng.choice(R, 200, replace=False), [0, 127, 128, R - 1]]))
    toks = np.unique(np.concatenate([rng.choice(T, 60, replace=False), [0, 255, 256, T - 1]]))
    _check(Y.cpu().numpy(), W16, X16, K, rows, toks)


@pytest.mark.parametrize("R,T", [(3584, 2048), (3544, 2000)])
def test_gemm_f16_last_wave_split(cuda_ready, R, T):
    # 224 tiles of 128 x 256 on 152 CTAs: the last 72 run as 144 tiles of 128 x 128
    # (ragged rows and tokens in the second case); every output is checked, and the
    # output starts as NaN so a tile left out shows
    import torch
    mq = cuda_ready
    K = 256
    W16, X16 = _gemm_case(R, K, T, seed=R + T)
    Y = torch.full((T, R), float("nan"), dtype=torch.float32, device="cuda")
    mq.gemm_f16(_dev(W16.view(np.float16)), _dev(X16.view(np.float16)), out=Y)
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    _check(Y.cpu().numpy(), W16, X16, K)


@pytest.mark.slow
def test_prefill_7b_ffn_gu_sampled(cuda_ready):
    # the 7B ffn_gu projection at 2K tokens, the pages' prefill size: the cache built on
    # the GPU (checked bit for bit on sampled rows), the GEMM checked on sampled outputs
    import torch
    mq = cuda_ready
    H, I, T = 3584, 18944, 2048
    W = synth.q4K_matrix(2 * I, H, seed=83, tag=synth.TAG_GU)
    x = synth.activation(H, T, seed=84)
    W16 = mq.dequant_q4K_f16(_dev(W), 2 * I, H)
    X16 = mq.convert_f32_f16(_dev(x))
    Y = mq.gemm_f16(W16, X16)
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    rng = np.random.default_rng(85)
    rows = np.unique(np.concatenate([rng.choice(2 * I, 48, replace=False), [0, 2 * I - 1]]))
    toks = np.unique(np.concatenate([rng.choice(T, 12, replace=False), [0, T - 1]]))
    w16 = W16[torch.from_numpy(rows).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(w16, oracle.dequant_q4K_f16(W[rows], H))
    x16 = X16.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(x16[toks], oracle.f32_to_f16_array(x[toks]))
    # the oracle on the sampled rows (their own cache rows) and tokens
    y_ref, Tm = oracle.gemm_f16(w16, x16, H, row_ids=np.arange(rows.size), tok_ids=toks)
    yg = Y.cpu().numpy()[np.ix_(toks, rows)]
    assert oracle.within_tolerance(yg, y_ref, Tm).all()
    del W16, X16, Y
    torch.cuda.empty_cache()
