"""q4_K x q8_0 matvec on the GPU against the oracle.

Bar: per-32-block int32 sums bit-exact (test export through the same device
code as the kernel); float outputs within |y - y_ref| <= 1e-3*T + 1e-5 with T
the oracle's sum of |per-block products|.
"""
import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth

pytestmark = pytest.mark.gpu


def _to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _check_y(y_gpu, W, xq_np, rows, K):
    y_ref, T = oracle.matvec(W, xq_np, rows, K)
    ok = oracle.within_tolerance(y_gpu, y_ref, T)
    if not ok.all():
        i = np.argwhere(~ok)[0]
        raise AssertionError(f"{(~ok).sum()} outside tolerance; first {tuple(i)}: gpu {y_gpu[tuple(i)]} "
                             f"ref {y_ref[tuple(i)]} T {T[tuple(i)]}")


SHAPES = [(1, 256), (7, 256), (33, 512), (300, 1024), (129, 1280), (64, 2304), (200, 3584),
          (77, 4864), (40, 18944), (1000, 256), (3, 8192)]


@pytest.mark.parametrize("rows,K", SHAPES)
@pytest.mark.parametrize("ncols", [1, 2, 8])
def test_matvec_parity_small(cuda_ready, variant, rows, K, ncols):
    import torch
    mq = cuda_ready
    if K * ncols > mq.MQ_MAX_K_TIMES_NCOLS:
        pytest.skip("beyond the staged-activation limit")
    W = synth.q4K_matrix(rows, K, seed=rows * 7 + K, tag=synth.TAG_W)
    x = synth.activation(K, ncols, seed=rows + K + ncols, tag=synth.TAG_X)
    xq_np = oracle.quantize_q8_0(x)
    Wd = _to_dev(W)
    # fp32 input, quantized inside the kernel
    y1, _ = mq.matvec_q4K_q8_0(Wd, rows, K, x=_to_dev(x))
    # pre-quantized q8_0 input
    y2, _ = mq.matvec_q4K_q8_0(Wd, rows, K, xq=_to_dev(xq_np))
    torch.cuda.synchronize()
    y1 = y1.cpu().numpy()
    y2 = y2.cpu().numpy()
    _check_y(y1, W, xq_np, rows, K)
    # both paths stage identical activations: identical bits
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("ncols", [1, 3, 4, 5, 6, 7])
def test_matvec_all_ncols(cuda_ready, variant, ncols):
    import torch
    mq = cuda_ready
    rows, K = 257, 3584
    W = synth.q4K_matrix(rows, K, seed=11, tag=synth.TAG_W)
    x = synth.activation(K, ncols, seed=12 + ncols, tag=synth.TAG_X)
    y, _ = mq.matvec_q4K_q8_0(_to_dev(W), rows, K, x=_to_dev(x))
    torch.cuda.synchronize()
    _check_y(y.cpu().numpy(), W, oracle.quantize_q8_0(x), rows, K)


@pytest.mark.parametrize("rows,K,ncols", [(5, 256, 1), (67, 3584, 1), (19, 18944, 2), (9, 1024, 8), (3, 4864, 3)])
def test_block_sums_bit_exact(cuda_ready, rows, K, ncols):
    import torch
    mq = cuda_ready
    W = synth.q4K_matrix(rows, K, seed=rows, tag=synth.TAG_W)
    x = synth.activation(K, ncols, seed=K, tag=synth.TAG_X)
    xq_np = oracle.quantize_q8_0(x)
    for kw in ({"x": _to_dev(x)}, {"xq": _to_dev(xq_np)}):
        sumi, sumq = mq.block_sums(_to_dev(W), rows, K, ncols=ncols, **kw)
        torch.cuda.synchronize()
        ri, rq = oracle.block_sums(W, xq_np, rows, K)
        assert np.array_equal(sumi.cpu().numpy(), ri)
        assert np.array_equal(sumq.cpu().numpy(), rq)


def test_xq_out_matches_quantizer(cuda_ready):
    import torch
    mq = cuda_ready
    rows, K, nc = 40, 3584, 2
    W = synth.q4K_matrix(rows, K, seed=1)
    x = synth.activation(K, nc, seed=2)
    xq_out = torch.zeros((nc, K // 32 * 34), dtype=torch.uint8, device="cuda")
    mq.matvec_q4K_q8_0(_to_dev(W), rows, K, x=_to_dev(x), xq_out=xq_out)
    torch.cuda.synchronize()
    assert np.array_equal(xq_out.cpu().numpy(), oracle.quantize_q8_0(x))


def test_deterministic_aa(cuda_ready, variant):
    # A/A control: the same call twice gives the same bits (no atomics, fixed reduction order)
    import torch
    mq = cuda_ready
    rows, K = 3584, 18944
    W = _to_dev(synth.q4K_matrix(rows, K, seed=5))
    x = _to_dev(synth.activation(K, 1, seed=6))
    y1, _ = mq.matvec_q4K_q8_0(W, rows, K, x=x)
    y2, _ = mq.matvec_q4K_q8_0(W, rows, K, x=x)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))


def test_y_ld_and_untouched_padding(cuda_ready):
    import torch
    mq = cuda_ready
    rows, K, nc = 100, 1024, 3
    W = synth.q4K_matrix(rows, K, seed=8)
    x = synth.activation(K, nc, seed=9)
    y = torch.full((nc, 128), 7.0, dtype=torch.float32, device="cuda")
    mq.matvec_q4K_q8_0(_to_dev(W), rows, K, x=_to_dev(x), y=y)
    torch.cuda.synchronize()
    yc = y.cpu().numpy()
    assert np.all(yc[:, rows:] == 7.0)
    _check_y(np.ascontiguousarray(yc[:, :rows]), W, oracle.quantize_q8_0(x), rows, K)


def test_descriptor_mismatch_is_reported_not_written(cuda_ready):
    import torch
    mq = cuda_ready
    rows, K = 64, 512
    W = _to_dev(synth.q4K_matrix(rows, K, seed=3))
    x = _to_dev(synth.activation(K, 1, seed=3))
    y = torch.full((1, rows), 5.0, dtype=torch.float32, device="cuda")
    d = mq.mv_desc(W, rows, K, y, x=x, ncols=1)
    dd = mq.upload_struct(d, W.device)
    assert mq.mq_read_device_status(0) == 0
    # the host says 32 rows, the device descriptor says 64: the kernel must refuse
    st = mq.mq_matvec_q4K_q8_0(dd.data_ptr(), 32, K, 1, torch.cuda.current_stream().cuda_stream)
    assert st == mq.MQ_OK
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) & mq.MQ_DEV_DESC_MISMATCH
    assert torch.all(y == 5.0)
    assert mq.mq_read_device_status(0) == 0


# ---- the workloads at full size ------------------------------------------------------------------

def test_matvec_512x1024_full(cuda_ready):
    import torch
    mq = cuda_ready
    case = synth.MATVEC_512x1024
    W, x = synth.matvec_case_inputs(case)
    y, _ = mq.matvec_q4K_q8_0(_to_dev(W), case.rows, case.K, x=_to_dev(x))
    torch.cuda.synchronize()
    _check_y(y.cpu().numpy(), W, oracle.quantize_q8_0(x), case.rows, case.K)


@pytest.mark.parametrize("K", synth.KSWEEP_KS)
def test_k_sweep_full(cuda_ready, variant, K):
    import torch
    mq = cuda_ready
    W, x = synth.ksweep_inputs(K)
    y, _ = mq.matvec_q4K_q8_0(_to_dev(W), synth.KSWEEP_ROWS, K, x=_to_dev(x))
    torch.cuda.synchronize()
    _check_y(y.cpu().numpy(), W, oracle.quantize_q8_0(x), synth.KSWEEP_ROWS, K)


def test_7b_down_matrix_full(cuda_ready, variant):
    # down projection of the 7B FFN: 3584 x 18944, every output row against the oracle
    import torch
    mq = cuda_ready
    W = synth.q4K_matrix(3584, 18944, seed=1, tag=synth.TAG_DOWN)
    x = synth.activation(18944, 1, seed=1, tag=synth.TAG_COLS)
    y, _ = mq.matvec_q4K_q8_0(_to_dev(W), 3584, 18944, x=_to_dev(x))
    torch.cuda.synchronize()
    _check_y(y.cpu().numpy(), W, oracle.quantize_q8_0(x), 3584, 18944)


def _device_plan(mq, rows, K, ncols):
    """The launch plan of this matvec on the current device, from the host planner."""
    import torch
    pr = torch.cuda.get_device_properties(torch.cuda.current_device())
    smem = getattr(pr, "shared_memory_per_block_optin", 0)
    l2 = getattr(pr, "L2_cache_size", 0)
    if not smem or not l2:
        pytest.skip("device properties for the planner not exposed by this torch")
    return mq.debug_plan_mv(mq.MQ_PLAN_MATVEC, rows, K, ncols, 0, num_sms=pr.multi_processor_count,
                            l2_bytes=l2, max_smem=smem)


# (rows, K, ncols) whose staged activation does not fit beside a ring of their
# rows: 8 and 4 columns on half-unit lanes (two parts), 6 columns on column
# groups (three parts), 3 columns on column groups (two parts)
K_SPLIT_CASES = [(200, 18944, 8), (200, 32256, 4), (200, 23808, 6), (200, 38912, 3)]


@pytest.mark.parametrize("rows,K,ncols", K_SPLIT_CASES)
def test_matvec_k_split_matches_oracle_and_exports_xq(cuda_ready, rows, K, ncols):
    """Columns x K too large to stage beside a ring of the CTA's rows: the matvec
    runs as a K split, one launch per part of every row, the later parts adding
    their sums to y.  The result stays within tolerance of the oracle, the fp32
    and q8_0 inputs give the same bits, and the q8_0 export of the activation
    (each part writes its range) is the whole activation, bit for bit."""
    import torch
    mq = cuda_ready
    plan = _device_plan(mq, rows, K, ncols)
    assert plan["variant"] == 1 and plan["ksplit"] > 1, plan
    W = synth.q4K_matrix(rows, K, seed=91 + ncols, tag=synth.TAG_W)
    x = synth.activation(K, ncols, seed=92 + ncols, tag=synth.TAG_X)
    xq_np = oracle.quantize_q8_0(x)
    Wd = _to_dev(W)
    xq_out = torch.zeros((ncols, K // 32 * 34), dtype=torch.uint8, device="cuda")
    y1, _ = mq.matvec_q4K_q8_0(Wd, rows, K, x=_to_dev(x), xq_out=xq_out)
    y2, _ = mq.matvec_q4K_q8_0(Wd, rows, K, xq=_to_dev(xq_np))
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    y1 = y1.cpu().numpy()
    _check_y(y1, W, xq_np, rows, K)
    assert np.array_equal(y1.view(np.uint32), y2.cpu().numpy().view(np.uint32))
    assert np.array_equal(xq_out.cpu().numpy(), xq_np.reshape(ncols, -1))


@pytest.mark.parametrize("K,ncols", [(131072, 1), (65536, 2)])
def test_matvec_k_split_long_rows(cuda_ready, K, ncols):
    """The longest rows the library takes (K * ncols up to its staged-activation
    limit) do not fit beside a ring in one launch either: one or two columns run
    as a K split of the whole-row kernels' two-column consumer."""
    import torch
    mq = cuda_ready
    rows = 37
    plan = _device_plan(mq, rows, K, ncols)
    assert plan["variant"] == 1 and plan["ksplit"] > 1, plan
    W = synth.q4K_matrix(rows, K, seed=K + ncols, tag=synth.TAG_W)
    x = synth.activation(K, ncols, seed=K + 1, tag=synth.TAG_X)
    xq_np = oracle.quantize_q8_0(x)
    Wd = _to_dev(W)
    y1, _ = mq.matvec_q4K_q8_0(Wd, rows, K, x=_to_dev(x))
    y2, _ = mq.matvec_q4K_q8_0(Wd, rows, K, xq=_to_dev(xq_np))
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    y1 = y1.cpu().numpy()
    _check_y(y1, W, xq_np, rows, K)
    assert np.array_equal(y1.view(np.uint32), y2.cpu().numpy().view(np.uint32))
