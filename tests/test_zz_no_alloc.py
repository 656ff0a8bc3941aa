"""mq_ffn_gu_silu_down_noalloc: the fused FFN on the library's own fixed
scratch.  Host checks run on the CPU; on the GPU its y must equal, bit for
bit, that of mq_ffn_gu_silu_down (caller scratch, same kernels) on two calls
in a row with different inputs, so the second call cannot pass on the first
call's leftovers.  Kept in a file of its own, collected after the others, so
that it runs both alone and after every other test of the session."""
import numpy as np
import pytest

from quantized_decode_matvec_gb300 import synth

RB = {3584: 14 * 144, 18944: 74 * 144}


def test_noalloc_host_checks(mq_lib):
    m = mq_lib
    f = m.mq_ffn_gu_silu_down_noalloc
    W_gu, W_down, x, y = 0x10000, 0x20000, 0x30000, 0x40000
    # h_q8 of the 7B FFN: 592 blocks of 34 bytes per column; 6 columns fit, 7 do not
    assert 6 * 592 * 34 <= m.MQ_NOALLOC_HQ8_MAX_BYTES < 7 * 592 * 34
    assert f(W_gu, W_down, x, 0, y, 3584, 18944, 7, 3584) == m.MQ_ERR_UNSUPPORTED
    assert f(W_gu, W_down, x, 0, y, 3584, 18944, 8, 3584) == m.MQ_ERR_UNSUPPORTED
    # the descriptor rules of mq_check_ffn_desc, before any device work
    assert f(W_gu, W_down, x, 0, y, 3584, 100, 1, 3584) == m.MQ_ERR_SHAPE
    assert f(W_gu, W_down, x, 0, y, 3584, 18944, 1, 3583) == m.MQ_ERR_SHAPE
    assert f(0, W_down, x, 0, y, 3584, 18944, 1, 3584) == m.MQ_ERR_INVALID_ARG
    assert f(W_gu, W_down, 0, 0, y, 3584, 18944, 1, 3584) == m.MQ_ERR_INVALID_ARG
    assert f(W_gu + 8, W_down, x, 0, y, 3584, 18944, 1, 3584) == m.MQ_ERR_ALIGN
    assert f(W_gu, W_down, x + 2, 0, y, 3584, 18944, 1, 3584) == m.MQ_ERR_ALIGN
    # no columns: nothing to do
    assert f(W_gu, W_down, x, 0, y, 3584, 18944, 0, 3584) == m.MQ_OK


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("H,I,ncols,use_xq", [(3584, 18944, 1, False), (3584, 18944, 6, False),
                                              (1024, 4864, 2, True), (512, 1024, 3, False)])
def test_noalloc_equals_caller_scratch(cuda_ready, H, I, ncols, use_xq):
    import torch
    mq = cuda_ready
    W_gu = _dev(synth.q4K_matrix(2 * I, H, seed=11, tag=1))
    W_down = _dev(synth.q4K_matrix(H, I, seed=11, tag=2))
    for call in range(2):
        x = _dev(synth.activation(H, ncols=ncols, seed=11, tag=3 + call))
        kw = {"xq": mq.quantize_q8_0(x)} if use_xq else {"x": x}
        ref = mq.ffn_gu_silu_down(W_gu, W_down, H, I, **kw)["y"]
        y = torch.full((ncols, H), float("nan"), dtype=torch.float32, device="cuda")
        mq.ffn_gu_silu_down_noalloc(W_gu, W_down, H, I, y=y, **kw)
        torch.cuda.synchronize()
        assert torch.isfinite(y).all(), f"call {call}"
        assert torch.equal(y, ref), f"call {call}: max |diff| {(y - ref).abs().max().item()}"
    assert mq.mq_read_device_status() == 0


@pytest.mark.gpu
def test_noalloc_strided_output_and_stream(cuda_ready):
    """y_ld > H leaves the gap untouched; the call runs on the given stream."""
    import torch
    mq = cuda_ready
    H, I, ncols, y_ld = 512, 1024, 2, 640
    W_gu = _dev(synth.q4K_matrix(2 * I, H, seed=12, tag=1))
    W_down = _dev(synth.q4K_matrix(H, I, seed=12, tag=2))
    x = _dev(synth.activation(H, ncols=ncols, seed=12, tag=3))
    ref = mq.ffn_gu_silu_down(W_gu, W_down, H, I, x=x)["y"]
    torch.cuda.synchronize()
    y = torch.full((ncols, y_ld), -7.0, dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())  # the fill above runs on the current stream
    with torch.cuda.stream(s):
        mq.ffn_gu_silu_down_noalloc(W_gu, W_down, H, I, x=x, y=y, stream=s)
    s.synchronize()
    assert torch.equal(y[:, :H], ref)
    assert (y[:, H:] == -7.0).all()
