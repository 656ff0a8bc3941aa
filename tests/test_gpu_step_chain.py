"""Chained decode steps and FFN-only stacks through mq_step.

A chained step is a real decode chain: the o projection reads the q|k|v
output, the FFN reads the o output and the next layer's q|k|v reads the FFN
output.  The persistent kernel passes those outputs between CTAs as tagged
records; the multi-kernel path orders them by kernel boundaries.  Both must
give the same bytes, and every phase must match the oracle on its own GPU
input (teacher-forced: the chain has no normalization, so its values drift
from layer to layer, and each phase is checked on the input it really read).
The weights' d and dmin are drawn smaller, with dmin large enough that the
weights' mean is about zero (synth d_scale, dmin_scale), so that a few layers
stay finite and of order one (checked beforehand by running the same chain on
the oracle).
"""
import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth

pytestmark = pytest.mark.gpu


def _weights(case, d_scale, ffn_only=False):
    """d_scale == 1: the workloads' draws; otherwise a chain's (mean about zero)."""
    import torch
    out, host = [], []
    for l in range(case.n_layers):
        w = synth.step_layer_weights(case, l, d_scale, dmin_scale=None if d_scale == 1.0 else 15 * d_scale)
        h = {"gu": w["gu"], "down": w["down"]}
        if not ffn_only:
            h["qkv"] = np.concatenate([w["q"], w["k"], w["v"]])
            h["o"] = w["o"]
        host.append(h)
        out.append({k: torch.from_numpy(v).cuda() for k, v in h.items()})
    return out, host


def _bufs(mq, case, wdev, chained, ffn_only=False, debug=True):
    qkv_rows = 0 if ffn_only else case.qkv_rows
    o_rows = 0 if ffn_only else case.H
    return mq.StepBuffers(wdev, case.H, case.I, qkv_rows, o_rows, case.q_rows, case.ncols, debug=debug,
                          chained=chained)


KEYS = ("y_qkv", "y_o", "y_ffn", "h_q8")


def _outputs(bufs):
    import torch
    torch.cuda.synchronize()
    return {k: getattr(bufs, k).cpu().numpy().copy() for k in KEYS}


def _feed(bufs, case, replay):
    import torch
    for l in range(case.n_layers):
        inp = synth.step_layer_inputs(case, l, replay)
        bufs.a[l].copy_(torch.from_numpy(inp["a"]))
        bufs.b[l].copy_(torch.from_numpy(inp["b"]))
        bufs.c[l].copy_(torch.from_numpy(inp["c"]))


def _same_bytes(x, y):
    for k in KEYS:
        assert np.array_equal(x[k].view(np.uint8), y[k].view(np.uint8)), k


def _check_chain_oracle(case, host, outs, first_input, ffn_only=False):
    """Every phase of every layer against the oracle on the input it read (teacher-forced)."""
    H, I = case.H, case.I
    x = first_input  # fp32 [ncols, K] read by the launch's first phase
    for l in range(case.n_layers):
        if not ffn_only:
            y_ref, T = oracle.matvec(host[l]["qkv"], oracle.quantize_q8_0(x), case.qkv_rows, H)
            assert oracle.within_tolerance(outs["y_qkv"][l], y_ref, T).all(), ("qkv", l)
            xb = outs["y_qkv"][l][:, :case.q_rows]
            y_ref, T = oracle.matvec(host[l]["o"], oracle.quantize_q8_0(xb), H, case.q_rows)
            assert oracle.within_tolerance(outs["y_o"][l], y_ref, T).all(), ("o", l)
            x = outs["y_o"][l]
        # the FFN: h_q8 against the oracle's chain on the FFN's input (codes may differ
        # only where h sits on a rounding edge), down teacher-forced on the kernel's h_q8
        _, hq_ref = oracle.ffn(host[l]["gu"], host[l]["down"], x, H, I)
        assert np.mean(outs["h_q8"][l] == hq_ref) > 0.99, ("h_q8", l)
        y_ref, T = oracle.matvec(host[l]["down"], outs["h_q8"][l], H, I)
        assert oracle.within_tolerance(outs["y_ffn"][l], y_ref, T).all(), ("down", l)
        assert np.isfinite(outs["y_ffn"][l]).all()
        x = outs["y_ffn"][l]


CHAIN_CASES = [
    (synth.StepCase("chain_small", 3, 512, 1024, 512, 128, 1, 31), 0.07),
    (synth.StepCase("chain_wide", 2, 3584, 4864, 3584, 512, 1, 32), 0.025),
    # two columns: q|k|v has as many rows as o has K (no k/v rows) so the chain keeps its stride
    (synth.StepCase("chain_ncols2", 2, 512, 1024, 512, 0, 2, 33), 0.06),
]


@pytest.mark.parametrize("case,d_scale", CHAIN_CASES, ids=[c.name for c, _ in CHAIN_CASES])
def test_chained_persistent_equals_multikernel_and_oracle(cuda_ready, case, d_scale):
    mq = cuda_ready
    wdev, host = _weights(case, d_scale)
    p = _bufs(mq, case, wdev, chained=True)
    q = _bufs(mq, case, wdev, chained=True)
    _feed(p, case, 0)
    _feed(q, case, 0)
    p.step()                                   # multi-kernel: kernel boundaries order the chain
    q.step(flags=mq.MQ_STEP_PERSISTENT)        # persistent: output records carry it
    x, y = _outputs(p), _outputs(q)
    assert mq.mq_read_device_status(0) == 0
    _same_bytes(x, y)
    assert np.array_equal(p.xq_a.cpu().numpy(), q.xq_a.cpu().numpy())
    assert np.array_equal(p.xq_b.cpu().numpy(), q.xq_b.cpu().numpy())
    a0 = synth.step_layer_inputs(case, 0, 0)["a"]
    _check_chain_oracle(case, host, y, a0)


def test_chained_graph_replays_byte_identical(cuda_ready):
    import torch
    from quantized_decode_matvec_gb300.graph import StepGraph
    mq = cuda_ready
    case, d_scale = CHAIN_CASES[0]
    wdev, host = _weights(case, d_scale)
    eager = _bufs(mq, case, wdev, chained=True)
    graphed = _bufs(mq, case, wdev, chained=True)
    g = StepGraph(graphed, flags=mq.MQ_STEP_PERSISTENT)
    assert g.captured, g.capture_error
    for r in range(4):
        _feed(eager, case, 50 + r)
        _feed(graphed, case, 50 + r)
        eager.step()
        g.run()
        torch.cuda.synchronize()
        _same_bytes(_outputs(eager), _outputs(graphed))
    assert mq.mq_read_device_status(0) == 0


FFN_CASES = [synth.StepCase("ffn_stack", 3, 1024, 4864, 0, 0, 1, 34),
             synth.StepCase("ffn_stack_ncols3", 2, 512, 1024, 0, 0, 3, 35)]


@pytest.mark.parametrize("chained", [False, True], ids=["independent", "chained"])
@pytest.mark.parametrize("case", FFN_CASES, ids=[c.name for c in FFN_CASES])
def test_ffn_only_stack(cuda_ready, case, chained):
    mq = cuda_ready
    d_scale = 0.04 if chained else 1.0
    wdev, host = _weights(case, d_scale, ffn_only=True)
    p = _bufs(mq, case, wdev, chained=chained, ffn_only=True, debug=False)
    q = _bufs(mq, case, wdev, chained=chained, ffn_only=True, debug=False)
    _feed(p, case, 0)
    _feed(q, case, 0)
    p.step()
    q.step(flags=mq.MQ_STEP_PERSISTENT)
    x, y = _outputs(p), _outputs(q)
    assert mq.mq_read_device_status(0) == 0
    _same_bytes(x, y)
    if chained:
        _check_chain_oracle(case, host, y, synth.step_layer_inputs(case, 0, 0)["c"], ffn_only=True)
    else:
        for l in range(case.n_layers):
            c = synth.step_layer_inputs(case, l, 0)["c"]
            _, hq_ref = oracle.ffn(host[l]["gu"], host[l]["down"], c, case.H, case.I)
            assert np.mean(y["h_q8"][l] == hq_ref) > 0.99
            y_ref, T = oracle.matvec(host[l]["down"], y["h_q8"][l], case.H, case.I)
            assert oracle.within_tolerance(y["y_ffn"][l], y_ref, T).all(), l


def _fill_outputs(bufs, value):
    bufs.outputs.fill_(value)
    bufs.h_q8.fill_(0x5A)


def test_persistent_rejects_chained_descriptors_without_the_flag(cuda_ready):
    # o.x == qkv.y (and the next layer's qkv.x == ffn.y) without MQ_STEP_CHAINED:
    # the kernel finds the overlap, records MQ_DEV_ALIAS and writes nothing
    import torch
    mq = cuda_ready
    case, d_scale = CHAIN_CASES[0]
    wdev, _ = _weights(case, d_scale)
    bufs = _bufs(mq, case, wdev, chained=True)
    _feed(bufs, case, 0)
    _fill_outputs(bufs, float("nan"))
    shape = mq.StepShape(case.n_layers, case.H, case.I, case.qkv_rows, case.H, case.q_rows, case.ncols,
                         mq.MQ_STEP_PERSISTENT, bufs.workspace.data_ptr())
    mq._check(mq.mq_step(bufs.table.data_ptr(), shape, torch.cuda.current_stream().cuda_stream), "mq_step")
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == mq.MQ_DEV_ALIAS
    assert torch.isnan(bufs.outputs).all()
    assert (bufs.h_q8 == 0x5A).all()
    # the same table with the flag runs
    bufs.step(flags=mq.MQ_STEP_PERSISTENT)
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == 0
    assert torch.isfinite(bufs.outputs).all()


def test_persistent_rejects_broken_chain(cuda_ready):
    # MQ_STEP_CHAINED on descriptors whose inputs are separate buffers: the chain
    # check records MQ_DEV_DESC_MISMATCH and nothing is written
    import torch
    mq = cuda_ready
    case, d_scale = CHAIN_CASES[0]
    wdev, _ = _weights(case, d_scale)
    bufs = _bufs(mq, case, wdev, chained=False)
    ws = torch.zeros(mq.mq_step_workspace_bytes(bufs.shape(mq.MQ_STEP_CHAINED)), dtype=torch.uint8,
                     device="cuda")
    _feed(bufs, case, 0)
    _fill_outputs(bufs, float("nan"))
    shape = mq.StepShape(case.n_layers, case.H, case.I, case.qkv_rows, case.H, case.q_rows, case.ncols,
                         mq.MQ_STEP_PERSISTENT | mq.MQ_STEP_CHAINED, ws.data_ptr())
    mq._check(mq.mq_step(bufs.table.data_ptr(), shape, torch.cuda.current_stream().cuda_stream), "mq_step")
    torch.cuda.synchronize()
    assert mq.mq_read_device_status(0) == mq.MQ_DEV_DESC_MISMATCH
    assert torch.isnan(bufs.outputs).all()
