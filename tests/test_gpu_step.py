"""The whole decode step of a layer stack (mq_step), eager and as a CUDA graph.

Graph tests follow "Part 4 . Lecture 08 -- Graph-Resident Decode": capture
plus at least seven replays, each with different inputs, each byte-compared
with an eager run on the same inputs (section 4); an A/A control before any
A/B (section 5); a deliberately frozen input that must go stale from replay 2
on (section 4); a failed capture that degrades to eager (section 3).
"""
import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth

pytestmark = pytest.mark.gpu

SMALL = synth.StepCase("step_small", n_layers=3, H=512, I=1024, q_rows=512, kv_rows=128, ncols=1, seed=5)


def _weights(case, device="cuda", concat_on_device=False):
    """Per-layer weights on the device and on the host.  With concat_on_device the
    q|k|v matrix is built on the GPU by mq_concat_rows (as the benchmark builds it)
    and checked byte for byte against the host concatenation."""
    import torch
    from quantized_decode_matvec_gb300 import mq
    out, host = [], []
    for l in range(case.n_layers):
        w = synth.step_layer_weights(case, l)
        qkv = np.concatenate([w["q"], w["k"], w["v"]])          # row concatenation q|k|v
        host.append({"qkv": qkv, "o": w["o"], "gu": w["gu"], "down": w["down"]})
        dev = {k: torch.from_numpy(v).to(device) for k, v in host[-1].items() if k != "qkv"}
        if concat_on_device:
            parts = [torch.from_numpy(w[n]).to(device) for n in ("q", "k", "v")]
            qkv_d = torch.empty(qkv.shape, dtype=torch.uint8, device=device)
            st = mq.mq_concat_rows(qkv_d.data_ptr(), [t.data_ptr() for t in parts],
                                   [case.q_rows, case.kv_rows, case.kv_rows], mq.MQ_TYPE_Q4_K, case.H,
                                   torch.cuda.current_stream().cuda_stream)
            assert st == mq.MQ_OK
            torch.cuda.synchronize()
            assert np.array_equal(qkv_d.cpu().numpy(), qkv), f"mq_concat_rows q|k|v, layer {l}"
            dev["qkv"] = qkv_d
            del parts
        else:
            dev["qkv"] = torch.from_numpy(qkv).to(device)
        out.append(dev)
    return out, host


def _inputs(case, replay):
    a = np.stack([synth.step_layer_inputs(case, l, replay)["a"] for l in range(case.n_layers)])
    b = np.stack([synth.step_layer_inputs(case, l, replay)["b"] for l in range(case.n_layers)])
    c = np.stack([synth.step_layer_inputs(case, l, replay)["c"] for l in range(case.n_layers)])
    return a, b, c


def _bufs(mq, case, wdev, debug=False):
    return mq.StepBuffers(wdev, case.H, case.I, case.qkv_rows, case.H, case.q_rows, case.ncols, debug=debug)


def _outputs(bufs):
    import torch
    torch.cuda.synchronize()
    return {k: getattr(bufs, k).cpu().numpy().copy() for k in ("y_qkv", "y_o", "y_ffn", "h_q8")}


def _set_inputs(bufs, a, b, c):
    import torch
    bufs.a.copy_(torch.from_numpy(a))
    bufs.b.copy_(torch.from_numpy(b))
    bufs.c.copy_(torch.from_numpy(c))


def _check_layer_oracle(case, host, outs, a, b, c, l, rows=None):
    """Layer l of a step against the oracle (sampled rows if given); FFN teacher-forced on h_q8."""
    H, I = case.H, case.I
    rs = lambda n: None if rows is None else np.sort(np.unique(np.concatenate([rows % n, [0, n - 1]])))
    for name, W, x, K, y in (("qkv", host[l]["qkv"], a[l], H, outs["y_qkv"][l]),
                             ("o", host[l]["o"], b[l], case.q_rows, outs["y_o"][l])):
        ids = rs(W.shape[0])
        y_ref, T = oracle.matvec(W, oracle.quantize_q8_0(x), W.shape[0], K, row_ids=ids)
        yg = y if ids is None else y[:, ids]
        assert oracle.within_tolerance(yg, y_ref, T).all(), (name, l)
    ids = rs(H)
    y_ref, T = oracle.matvec(host[l]["down"], outs["h_q8"][l], H, I, row_ids=ids)
    yg = outs["y_ffn"][l] if ids is None else outs["y_ffn"][l][:, ids]
    assert oracle.within_tolerance(yg, y_ref, T).all(), ("down", l)


def test_step_small_eager_matches_oracle(cuda_ready, variant):
    mq = cuda_ready
    wdev, host = _weights(SMALL)
    bufs = _bufs(mq, SMALL, wdev, debug=True)
    a, b, c = _inputs(SMALL, 0)
    _set_inputs(bufs, a, b, c)
    bufs.step()
    outs = _outputs(bufs)
    for l in range(SMALL.n_layers):
        _check_layer_oracle(SMALL, host, outs, a, b, c, l)
        assert np.array_equal(bufs.xq_a[l].cpu().numpy(), oracle.quantize_q8_0(a[l]))
        # h_q8 against the whole oracle FFN chain: codes may differ only where h sits on a rounding edge
        _, hq_ref = oracle.ffn(host[l]["gu"], host[l]["down"], c[l], SMALL.H, SMALL.I)
        assert np.mean(outs["h_q8"][l] == hq_ref) > 0.99


def test_step_graph_replays_byte_identical(cuda_ready, variant):
    import torch
    from quantized_decode_matvec_gb300.graph import StepGraph
    mq = cuda_ready
    wdev, host = _weights(SMALL)
    eager = _bufs(mq, SMALL, wdev)
    graphed = _bufs(mq, SMALL, wdev)
    g = StepGraph(graphed)
    assert g.captured, g.capture_error
    # A/A first: eager vs eager on the same inputs
    a, b, c = _inputs(SMALL, 100)
    _set_inputs(eager, a, b, c)
    eager.step()
    first = _outputs(eager)
    eager.step()
    again = _outputs(eager)
    for k in first:
        assert np.array_equal(first[k], again[k])
    # capture + 7 replays with fresh inputs each, byte-compared with eager
    for r in range(8):
        a, b, c = _inputs(SMALL, r)
        _set_inputs(eager, a, b, c)
        eager.step()
        e = _outputs(eager)
        _set_inputs(graphed, a, b, c)
        g.run()
        torch.cuda.synchronize()
        gr = _outputs(graphed)
        for k in e:
            assert np.array_equal(e[k].view(np.uint8), gr[k].view(np.uint8)), (r, k)
        if r in (0, 7):
            for l in (0, SMALL.n_layers - 1):
                _check_layer_oracle(SMALL, host, gr, a, b, c, l)


def test_frozen_input_goes_stale_from_replay_2(cuda_ready):
    # Negative control: a runner that captures its input copy from the staging slot
    # chosen at capture time.  Replay 1 reuses that slot and is right; from replay 2
    # the inputs sit in other slots and the graph keeps reading the frozen one.
    import torch
    mq = cuda_ready
    wdev, host = _weights(SMALL)
    bufs = _bufs(mq, SMALL, wdev)
    eager = _bufs(mq, SMALL, wdev)
    slots = [torch.empty((3,) + tuple(bufs.a.shape), dtype=torch.float32, device="cuda") for _ in range(4)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        bufs.step(s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    frozen = slots[0]
    with torch.cuda.graph(g, stream=s):
        bufs.a.copy_(frozen[0])
        bufs.b.copy_(frozen[1])
        bufs.c.copy_(frozen[2])
        bufs.step(s)
    mism = []
    for r in range(4):
        a, b, c = _inputs(SMALL, r)
        slot = slots[r % len(slots)] if r > 0 else slots[0]
        slot[0].copy_(torch.from_numpy(a))
        slot[1].copy_(torch.from_numpy(b))
        slot[2].copy_(torch.from_numpy(c))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        _set_inputs(eager, a, b, c)
        eager.step()
        e = _outputs(eager)
        gr = _outputs(bufs)
        mism.append(not np.array_equal(e["y_ffn"], gr["y_ffn"]))
    assert mism == [False, True, True, True]


def test_capture_failure_falls_back_to_eager(cuda_ready):
    import torch
    from quantized_decode_matvec_gb300.graph import StepGraph
    mq = cuda_ready
    wdev, host = _weights(SMALL)
    bufs = _bufs(mq, SMALL, wdev)
    # a synchronizing host call inside the capture window is illegal during capture
    g = StepGraph(bufs, capture_hook=lambda: torch.cuda.synchronize())
    assert not g.captured and g.capture_error
    a, b, c = _inputs(SMALL, 3)
    _set_inputs(bufs, a, b, c)
    g.run()
    outs = _outputs(bufs)
    _check_layer_oracle(SMALL, host, outs, a, b, c, 0)
    _check_layer_oracle(SMALL, host, outs, a, b, c, SMALL.n_layers - 1)


def test_step_pdl_matches_plain(cuda_ready, variant):
    mq = cuda_ready
    wdev, host = _weights(SMALL)
    p = _bufs(mq, SMALL, wdev)
    q = _bufs(mq, SMALL, wdev)
    a, b, c = _inputs(SMALL, 4)
    _set_inputs(p, a, b, c)
    _set_inputs(q, a, b, c)
    p.step()
    q.step(flags=mq.MQ_STEP_PDL)
    x, y = _outputs(p), _outputs(q)
    for k in x:
        assert np.array_equal(x[k].view(np.uint8), y[k].view(np.uint8)), k


# every column count's consumer form in the persistent kernel: 1-2 columns keep
# the activation in registers (2 columns: the two-column register path), 3-4
# read it from shared memory per row pair, 5-8 run on column lanes
PERSISTENT_CASES = [SMALL, synth.StepCase("step_tiny", 2, 256, 256, 256, 256, 1, 6),
                    synth.StepCase("step_ncols2", 2, 1024, 1536, 1024, 256, 2, 10),
                    synth.StepCase("step_ncols3", 2, 512, 768, 512, 128, 3, 7),
                    synth.StepCase("step_ncols4", 2, 512, 1024, 512, 128, 4, 11),
                    synth.StepCase("step_ncols5", 2, 512, 768, 512, 128, 5, 12),
                    synth.StepCase("step_ncols8", 2, 768, 1024, 768, 128, 8, 13),
                    synth.StepCase("step_ncols2_long", 1, 3584, 4864, 3584, 512, 2, 14)]


@pytest.mark.parametrize("case", PERSISTENT_CASES, ids=[c.name for c in PERSISTENT_CASES])
def test_persistent_step_bit_identical_to_multikernel(cuda_ready, case):
    mq = cuda_ready
    wdev, host = _weights(case)
    p = _bufs(mq, case, wdev, debug=True)
    q = _bufs(mq, case, wdev, debug=True)
    a, b, c = _inputs(case, 9)
    _set_inputs(p, a, b, c)
    _set_inputs(q, a, b, c)
    p.step()
    q.step(flags=mq.MQ_STEP_PERSISTENT)
    x, y = _outputs(p), _outputs(q)
    assert mq.mq_read_device_status(0) == 0
    for k in x:
        assert np.array_equal(x[k].view(np.uint8), y[k].view(np.uint8)), k
    assert np.array_equal(p.xq_a.cpu().numpy(), q.xq_a.cpu().numpy())
    for l in range(case.n_layers):
        _check_layer_oracle(case, host, y, a, b, c, l)


def test_persistent_step_graph_replays(cuda_ready):
    import torch
    from quantized_decode_matvec_gb300.graph import StepGraph
    mq = cuda_ready
    wdev, host = _weights(SMALL)
    eager = _bufs(mq, SMALL, wdev)
    graphed = _bufs(mq, SMALL, wdev)
    g = StepGraph(graphed, flags=mq.MQ_STEP_PERSISTENT)
    assert g.captured, g.capture_error
    for r in range(8):
        a, b, c = _inputs(SMALL, 20 + r)
        _set_inputs(eager, a, b, c)
        eager.step()
        e = _outputs(eager)
        _set_inputs(graphed, a, b, c)
        g.run()
        torch.cuda.synchronize()
        gr = _outputs(graphed)
        for k in e:
            assert np.array_equal(e[k].view(np.uint8), gr[k].view(np.uint8)), (r, k)
    assert mq.mq_read_device_status(0) == 0


@pytest.mark.slow
def test_step_7b_full_size_sampled(cuda_ready):
    # The 28-layer 7B-class step at full size exactly as the benchmark runs it:
    # q|k|v built on the device by mq_concat_rows, the persistent kernel captured
    # as one CUDA graph and replayed.  Every layer of every replay is checked
    # against the oracle on sampled rows (the FFN teacher-forced on the kernel's
    # h_q8), and the PDL multi-kernel graph gives the same bytes.
    import torch
    from quantized_decode_matvec_gb300.graph import StepGraph
    mq = cuda_ready
    case = synth.STEP_7B
    wdev, host = _weights(case, concat_on_device=True)
    bufs = _bufs(mq, case, wdev)
    multi = _bufs(mq, case, wdev)
    g = StepGraph(bufs, flags=mq.MQ_STEP_PERSISTENT)   # the benchmark's default launch mode
    assert g.captured, g.capture_error
    gp = StepGraph(multi, flags=mq.MQ_STEP_PDL)
    assert gp.captured, gp.capture_error
    rng = np.random.default_rng(0)
    rows = rng.choice(1 << 20, 48, replace=False)
    for r in (0, 1, 2):
        a, b, c = _inputs(case, r)
        _set_inputs(bufs, a, b, c)
        g.run()
        outs = _outputs(bufs)
        for l in range(case.n_layers):
            _check_layer_oracle(case, host, outs, a, b, c, l, rows=rows)
        _set_inputs(multi, a, b, c)
        gp.run()
        m = _outputs(multi)
        for k in outs:
            assert np.array_equal(outs[k].view(np.uint8), m[k].view(np.uint8)), (r, k)
    assert mq.mq_read_device_status(0) == 0
    del wdev, bufs, multi, g, gp
    torch.cuda.empty_cache()


def test_step_graph_with_host_io(cuda_ready):
    # the input copy, the persistent step and the output copy captured as one
    # graph: each replay reads the pinned inputs as they are at replay time and
    # leaves the outputs in pinned host memory, byte-identical to an eager step
    import torch
    from quantized_decode_matvec_gb300.graph import PinnedFeeder, StepGraph
    mq = cuda_ready
    wdev, host = _weights(SMALL)
    eager = _bufs(mq, SMALL, wdev)
    graphed = _bufs(mq, SMALL, wdev)
    feeder = PinnedFeeder(graphed)
    host_out = torch.empty(graphed.outputs.shape, dtype=torch.float32, pin_memory=True)
    g = StepGraph(graphed, flags=mq.MQ_STEP_PERSISTENT, io=(feeder.inputs, host_out))
    assert g.captured, g.capture_error
    for r in range(3):
        a, b, c = _inputs(SMALL, 40 + r)
        feeder.load(a, b, c)
        g.run()
        g.stream.synchronize()
        _set_inputs(eager, a, b, c)
        eager.step(flags=mq.MQ_STEP_PERSISTENT)
        torch.cuda.synchronize()
        assert np.array_equal(host_out.numpy().view(np.uint8), eager.outputs.cpu().numpy().view(np.uint8)), r
    assert mq.mq_read_device_status(0) == 0


def test_step_outputs_through_pinned_readback(cuda_ready):
    # the step's outputs read back through the self-held pinned buffer: a first
    # read into a buffer sized for it, then a read larger than that buffer
    # (5.6 MB against 4 MiB), which grows it; every read byte-identical to .cpu()
    import torch
    from quantized_decode_matvec_gb300.graph import PinnedReadback
    mq = cuda_ready
    wdev, host = _weights(SMALL)
    bufs = _bufs(mq, SMALL, wdev)
    _set_inputs(bufs, *_inputs(SMALL, 77))
    bufs.step(flags=mq.MQ_STEP_PERSISTENT)
    torch.cuda.synchronize()
    rb = PinnedReadback()
    out = rb.read(bufs.outputs)
    assert rb.capacity == PinnedReadback.MIN_BYTES and rb._buf.is_pinned() and rb.fallbacks == 0
    assert np.array_equal(out.numpy().view(np.uint8), bufs.outputs.cpu().numpy().view(np.uint8))
    big = torch.randint(-2**31, 2**31 - 1, (1_400_000,), dtype=torch.int32, device="cuda")
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    got = rb.read(big, stream=st)
    assert rb.capacity == 5_600_000 and rb.allocations == 2 and rb._buf.is_pinned()
    assert torch.equal(got, big.cpu())
    assert mq.mq_read_device_status(0) == 0
