"""Failure detection without a GPU fault.

The bulk-copy ring kernels bound every wait on their copy pipeline, and the
persistent step kernel every wait at its dependency points.  A
test-only setting makes the producer withhold each CTA's last tile, so the
consumers' waits run out (a flag that nothing ever sets): the kernel must
report MQ_DEV_TIMEOUT through the device status word, leave its output
untouched and return, and the context must stay usable for the next call.
"""
import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports(cuda_ready):
    import torch
    mq = cuda_ready
    rows, K = 3584, 3584          # planned on the ring kernels
    W = torch.from_numpy(synth.q4K_matrix(rows, K, seed=4)).cuda()
    x_np = synth.activation(K, 1, seed=4)
    x = torch.from_numpy(x_np).cuda()
    y = torch.full((1, rows), 3.0, dtype=torch.float32, device="cuda")
    assert mq.mq_read_device_status(0) == 0
    assert mq.mq_debug_set_fault(mq.MQ_FAULT_WITHHOLD_TILE) == mq.MQ_OK
    try:
        mq.matvec_q4K_q8_0(W, rows, K, x=x, y=y)
        torch.cuda.synchronize()                     # returns: the waits are bounded
    finally:
        assert mq.mq_debug_set_fault(mq.MQ_FAULT_NONE) == mq.MQ_OK
    assert mq.mq_read_device_status(0) & mq.MQ_DEV_TIMEOUT
    assert torch.all(y == 3.0)                       # nothing written
    # the context is still healthy: the same call now succeeds and matches the oracle
    y2, _ = mq.matvec_q4K_q8_0(W, rows, K, x=x)
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    y_ref, T = oracle.matvec(W.cpu().numpy(), oracle.quantize_q8_0(x_np), rows, K)
    assert oracle.within_tolerance(y2.cpu().numpy(), y_ref, T).all()


def test_fault_setter_rejects_unknown(cuda_ready):
    mq = cuda_ready
    assert mq.mq_debug_set_fault(7) == mq.MQ_ERR_INVALID_ARG
    assert mq.mq_debug_set_variant(7) == mq.MQ_ERR_INVALID_ARG


@pytest.mark.parametrize("fault", ["records", "count"])
def test_persistent_step_dependency_wait_runs_out_and_reports(cuda_ready, fault):
    # the persistent step's dependency waits are bounded too: with the last CTA's h
    # records withheld (every CTA's down phase runs out of time), or its phases never
    # added to the phase counter (every CTA's wait for the first phase's end runs out),
    # the abort word stops the launch, and the next step runs normally
    import torch
    mq = cuda_ready
    case = synth.StepCase("step_fault", 2, 512, 1024, 512, 128, 1, 11)
    wdev = []
    for l in range(case.n_layers):
        w = synth.step_layer_weights(case, l)
        wdev.append({"qkv": torch.from_numpy(np.concatenate([w["q"], w["k"], w["v"]])).cuda(),
                     "o": torch.from_numpy(w["o"]).cuda(), "gu": torch.from_numpy(w["gu"]).cuda(),
                     "down": torch.from_numpy(w["down"]).cuda()})
    bufs = [mq.StepBuffers(wdev, case.H, case.I, case.qkv_rows, case.H, case.q_rows, 1) for _ in range(2)]
    for b in bufs:
        for l in range(case.n_layers):
            inp = synth.step_layer_inputs(case, l, 3)
            b.a[l].copy_(torch.from_numpy(inp["a"]))
            b.b[l].copy_(torch.from_numpy(inp["b"]))
            b.c[l].copy_(torch.from_numpy(inp["c"]))
    assert mq.mq_read_device_status(0) == 0
    code = mq.MQ_FAULT_WITHHOLD_RECORDS if fault == "records" else mq.MQ_FAULT_WITHHOLD_COUNT
    assert mq.mq_debug_set_fault(code) == mq.MQ_OK
    try:
        bufs[0].step(flags=mq.MQ_STEP_PERSISTENT)
        torch.cuda.synchronize()                     # returns: every wait is bounded
    finally:
        assert mq.mq_debug_set_fault(mq.MQ_FAULT_NONE) == mq.MQ_OK
    assert mq.mq_read_device_status(0) & mq.MQ_DEV_TIMEOUT
    # the context is still healthy: the persistent step now matches the multi-kernel step bit for bit
    bufs[0].step(flags=mq.MQ_STEP_PERSISTENT)
    bufs[1].step()
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    for k in ("y_qkv", "y_o", "y_ffn", "h_q8"):
        x, y = getattr(bufs[0], k).cpu().numpy(), getattr(bufs[1], k).cpu().numpy()
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8)), k
