"""mq_concat_rows on the device: the row concatenation that builds ffn_gu (gate
rows, then up rows: "04 . 8o -- Killing the CPU stall at decode start",
sections 1 and 3.1) and the q|k|v projection, at the 7B-class shapes the
benchmark builds.  The device result must equal the host concatenation of the
same bytes, byte for byte; the preconditions of section 3.2 are checked on
the host before any copy."""
import numpy as np
import pytest

from quantized_decode_matvec_gb300 import synth

pytestmark = pytest.mark.gpu


def _concat_dev(mq, parts, rows, ttype, ne0):
    import torch
    dev = [torch.from_numpy(np.ascontiguousarray(p)).cuda() for p in parts]
    out = torch.full((sum(rows), parts[0].shape[1]), 0xA5, dtype=torch.uint8, device="cuda")
    st = mq.mq_concat_rows(out.data_ptr(), [t.data_ptr() for t in dev], rows, ttype, ne0,
                           torch.cuda.current_stream().cuda_stream)
    assert st == mq.MQ_OK, mq.status_string(st)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_concat_qkv_7b(cuda_ready):
    mq = cuda_ready
    case = synth.STEP_7B
    w = synth.step_layer_weights(case, 3)
    parts = [w["q"], w["k"], w["v"]]
    rows = [case.q_rows, case.kv_rows, case.kv_rows]
    got = _concat_dev(mq, parts, rows, mq.MQ_TYPE_Q4_K, case.H)
    assert np.array_equal(got, np.concatenate(parts))


def test_concat_ffn_gu_7b(cuda_ready):
    mq = cuda_ready
    H, I = synth.FFN_7B.H, synth.FFN_7B.I
    gate = synth.q4K_matrix(I, H, seed=21, tag=synth.TAG_GU)
    up = synth.q4K_matrix(I, H, seed=22, tag=synth.TAG_GU)
    got = _concat_dev(mq, [gate, up], [I, I], mq.MQ_TYPE_Q4_K, H)
    assert np.array_equal(got[:I], gate) and np.array_equal(got[I:], up)


@pytest.mark.parametrize("wtype,ttype_name", [("q4_0", "MQ_TYPE_Q4_0"), ("q8_0", "MQ_TYPE_Q8_0")])
def test_concat_other_types(cuda_ready, wtype, ttype_name):
    mq = cuda_ready
    K = 1024
    parts = [synth.wq_matrix(wtype, r, K, seed=30 + r) for r in (96, 1, 33)]
    got = _concat_dev(mq, parts, [96, 1, 33], getattr(mq, ttype_name), K)
    assert np.array_equal(got, np.concatenate(parts))


def test_concat_empty_part(cuda_ready):
    # a tensor of zero rows contributes nothing (a null pointer is allowed for it)
    import torch
    mq = cuda_ready
    K = 512
    a = synth.q4K_matrix(5, K, seed=40)
    b = synth.q4K_matrix(7, K, seed=41)
    ad, bd = (torch.from_numpy(t).cuda() for t in (a, b))
    out = torch.zeros((12, a.shape[1]), dtype=torch.uint8, device="cuda")
    st = mq.mq_concat_rows(out.data_ptr(), [ad.data_ptr(), 0, bd.data_ptr()], [5, 0, 7], mq.MQ_TYPE_Q4_K, K,
                           torch.cuda.current_stream().cuda_stream)
    assert st == mq.MQ_OK
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), np.concatenate([a, b]))
