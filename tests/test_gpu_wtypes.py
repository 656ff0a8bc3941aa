"""The matvec for q4_0 and q8_0 weights against the oracle: y within the
stated tolerance |y - y_ref| <= 1e-3 * sum|terms| + 1e-5 (terms: the
per-block products the oracle sums), on shapes that span several tiles
with ragged rows, 1..8 columns, fp32 and pre-quantized activations, and the
full-size shapes on sampled rows."""
import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth

pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-3, 1e-5


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check(y, yr, T):
    err = np.abs(y.astype(np.float64) - yr)
    bound = TOL_REL * T + TOL_ABS
    assert np.all(err <= bound), f"max err/bound {np.max(err / bound):.3g}"


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0"])
@pytest.mark.parametrize("rows,K,ncols", [(1, 256, 1), (37, 1024, 1), (300, 3584, 1), (1000, 4096, 2),
                                          (77, 512, 3), (129, 2048, 8), (4608, 3584, 1)])
def test_matches_oracle(cuda_ready, wtype, rows, K, ncols):
    import torch
    mq = cuda_ready
    W = synth.wq_matrix(wtype, rows, K, seed=rows + K)
    x = synth.activation(K, ncols, seed=rows + K + 1)
    y, _ = mq.matvec_w(wtype, _dev(W), rows, K, x=_dev(x))
    torch.cuda.synchronize()
    yr, T = oracle.matvec_w(wtype, W, oracle.quantize_q8_0(x), rows, K)
    _check(y.cpu().numpy(), yr, T)


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0"])
def test_prequantized_input_equals_fp32_input(cuda_ready, wtype):
    import torch
    mq = cuda_ready
    rows, K = 513, 4096
    W = _dev(synth.wq_matrix(wtype, rows, K, seed=31))
    x = _dev(synth.activation(K, 2, seed=32))
    y1, _ = mq.matvec_w(wtype, W, rows, K, x=x)
    y2, _ = mq.matvec_w(wtype, W, rows, K, xq=mq.quantize_q8_0(x))
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("wtype", ["q4_0", "q8_0"])
@pytest.mark.parametrize("rows,K", [(37888, 3584), (4096, 18944)])
def test_full_size_sampled_rows(cuda_ready, wtype, rows, K):
    import torch
    mq = cuda_ready
    W = synth.wq_matrix(wtype, rows, K, seed=41)
    x = synth.activation(K, 1, seed=42)
    y, _ = mq.matvec_w(wtype, _dev(W), rows, K, x=_dev(x))
    torch.cuda.synchronize()
    ids = np.unique(np.concatenate([np.arange(8), rows - 1 - np.arange(8),
                                    np.random.default_rng(0).integers(0, rows, 48)]))
    yr, T = oracle.matvec_w(wtype, W, oracle.quantize_q8_0(x), rows, K, row_ids=ids)
    _check(y.cpu().numpy()[:, ids], yr, T)


def test_edge_shapes_and_errors(cuda_ready):
    import torch
    mq = cuda_ready
    W = _dev(synth.wq_matrix("q4_0", 4, 256, seed=5))
    x = _dev(synth.activation(256, 1, seed=5))
    # no rows / no columns: nothing to do
    assert mq.mq_matvec_q4_0_q8_0(0, 0, 256, 1) == mq.MQ_OK
    assert mq.mq_matvec_q8_0_q8_0(0, 4, 256, 0) == mq.MQ_OK
    # K must be a multiple of 256
    assert mq.mq_matvec_q4_0_q8_0(0, 4, 96, 1) == mq.MQ_ERR_SHAPE
    y, _ = mq.matvec_w("q4_0", W, 4, 256, x=x)
    torch.cuda.synchronize()
    yr, T = oracle.matvec_w("q4_0", W.cpu().numpy(), oracle.quantize_q8_0(x.cpu().numpy()), 4, 256)
    _check(y.cpu().numpy(), yr, T)
    assert mq.mq_read_device_status() == 0
