"""The q4_K x q8_0 matmul for more columns on the tensor cores ("07 . R3 --
Small-model per-token overhead", section 5: MMQ) against the oracle.

Bars: the q8_0 codes it quantizes are bit-exact (xq_out); float outputs are
within |y - y_ref| <= 1e-3 * T + 1e-5 of the oracle's fp64 matvec, T the sum
of the per-block products' magnitudes, on every row at small sizes and on
sampled rows at the 7B shapes; fp32 input and pre-quantized input give the
same bits.
"""
import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check(y, W, xq, rows, K, row_ids=None):
    y_ref, T = oracle.matvec(W, xq, rows, K, row_ids=row_ids)
    yg = y if row_ids is None else y[:, row_ids]
    ok = oracle.within_tolerance(yg, y_ref, T)
    if not ok.all():
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError(f"{(~ok).sum()} outside tolerance; first {i}: gpu {yg[i]} ref {y_ref[i]} T {T[i]}")


# one tile / one step; ragged rows and columns; many steps; split K (few row tiles); N = 48 and 64
SHAPES = [(128, 256, 16), (300, 1024, 9), (256, 3584, 32), (520, 4864, 17), (3584, 3584, 64), (1000, 18944, 48),
          (64, 512, 64)]


@pytest.mark.parametrize("rows,K,ncols", SHAPES)
def test_mmq_parity(cuda_ready, rows, K, ncols):
    import torch
    mq = cuda_ready
    W = synth.q4K_matrix(rows, K, seed=rows + K + ncols)
    x = synth.activation(K, ncols, seed=rows * 7 + ncols)
    xq = oracle.quantize_q8_0(x)
    Wd = _dev(W)
    xq_out = torch.zeros((ncols, K // 32 * 34), dtype=torch.uint8, device="cuda")
    y1, _, ws = mq.mmq_q4K_q8_0(Wd, rows, K, x=_dev(x), xq_out=xq_out)
    y2, _, _ = mq.mmq_q4K_q8_0(Wd, rows, K, xq=_dev(xq), workspace=ws)
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    assert np.array_equal(xq_out.cpu().numpy(), xq)
    y1, y2 = y1.cpu().numpy(), y2.cpu().numpy()
    if rows * K * ncols <= 80_000_000:
        _check(y1, W, xq, rows, K)
    else:
        rng = np.random.default_rng(rows)
        ids = np.unique(np.concatenate([rng.choice(rows, 64, replace=False), [0, 127, 128, rows - 1]]))
        _check(y1, W, xq, rows, K, row_ids=ids)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


@pytest.mark.slow
@pytest.mark.parametrize("which,ncols", [("gu", 16), ("down", 64)])
def test_mmq_7b_ffn_shapes_sampled(cuda_ready, which, ncols):
    import torch
    mq = cuda_ready
    H, I = synth.FFN_7B.H, synth.FFN_7B.I
    rows, K = (2 * I, H) if which == "gu" else (H, I)
    W = synth.q4K_matrix(rows, K, seed=95, tag=synth.TAG_GU if which == "gu" else synth.TAG_DOWN)
    x = synth.activation(K, ncols, seed=96)
    xq = oracle.quantize_q8_0(x)
    y, _, _ = mq.mmq_q4K_q8_0(_dev(W), rows, K, x=_dev(x))
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    rng = np.random.default_rng(97)
    ids = np.unique(np.concatenate([rng.choice(rows, 48, replace=False), [0, rows - 1]]))
    _check(y.cpu().numpy(), W, xq, rows, K, row_ids=ids)


def test_mmq_strided_output_and_small_workspace(cuda_ready):
    import torch
    mq = cuda_ready
    rows, K, ncols, y_ld = 200, 512, 20, 256
    W = synth.q4K_matrix(rows, K, seed=98)
    x = synth.activation(K, ncols, seed=99)
    y = torch.full((ncols, y_ld), -3.0, dtype=torch.float32, device="cuda")
    mq.mmq_q4K_q8_0(_dev(W), rows, K, x=_dev(x), y=y)
    torch.cuda.synchronize()
    yn = y.cpu().numpy()
    _check(yn[:, :rows], W, oracle.quantize_q8_0(x), rows, K)
    assert (yn[:, rows:] == -3.0).all()
    # a workspace one byte short is refused before any launch
    need = mq.mq_mmq_workspace_bytes(rows, K, ncols)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    d = mq.upload_struct(mq.mv_desc(_dev(W), rows, K, y, x=_dev(x), ncols=ncols, y_ld=y_ld), y.device)
    assert mq.mq_mmq_q4K_q8_0(d.data_ptr(), rows, K, ncols, ws.data_ptr(), need - 1) == mq.MQ_ERR_INVALID_ARG
    assert mq.mq_mmq_q4K_q8_0(d.data_ptr(), rows, K, 65, ws.data_ptr(), need) == mq.MQ_ERR_SHAPE
