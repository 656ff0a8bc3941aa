"""Fused FFN (ffn_gu matvec -> SiLU*mul -> q8_0 -> down) against the oracle.

The chain cannot be bit-exact end to end (h comes from float sums and exp),
so parity is checked stage by stage with teacher forcing:
 (i)   g|u from the kernel vs the oracle matvec of ffn_gu, float tolerance;
 (ii)  the kernel's h vs the oracle's SiLU(g)*u of the kernel's own g, u,
       within 1e-6*|h| + 1e-7 (fp32 exp/div/mul rounding);
 (iii) the kernel's h_q8 bit-exact vs the oracle's q8_0 of the kernel's h;
 (iv)  y vs the oracle matvec of W_down with the kernel's h_q8, float tolerance.
Small cases also compare end to end with the pure-oracle chain, widening the
bound by the effect of every q8 code of h that differs between the chains.
"""
import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth
from tests.q4k_layout import dequant_q8, dequant_rows

pytestmark = pytest.mark.gpu


def _to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run(mq, W_gu, W_down, x, H, I, use_xq=False):
    import torch
    kw = {"xq": _to_dev(oracle.quantize_q8_0(x))} if use_xq else {"x": _to_dev(x)}
    out = mq.ffn_gu_silu_down(_to_dev(W_gu), _to_dev(W_down), H, I, debug=True, **kw)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items() if k != "desc"}


def _stagewise(out, W_gu, W_down, x, H, I, gu_rows=None, down_rows=None):
    nc = x.shape[0]
    xq = oracle.quantize_q8_0(x)
    # (i) g|u
    ids = None if gu_rows is None else np.asarray(gu_rows)
    gu_ref, T = oracle.matvec(W_gu, xq, 2 * I, H, row_ids=ids)
    gu_gpu = out["gu"] if ids is None else out["gu"][:, ids]
    assert oracle.within_tolerance(gu_gpu, gu_ref, T).all()
    # (ii) h from the kernel's own g, u
    g = out["gu"][:, :I].astype(np.float64)
    u = out["gu"][:, I:].astype(np.float64)
    h_ref = oracle.silu_mul(g, u)
    assert np.all(np.abs(out["h"] - h_ref) <= 1e-6 * np.abs(h_ref) + 1e-7)
    # (iii) h_q8 bit-exact from the kernel's h
    assert np.array_equal(out["h_q8"], oracle.quantize_q8_0(out["h"]))
    # (iv) y from the kernel's h_q8
    ids = None if down_rows is None else np.asarray(down_rows)
    y_ref, T = oracle.matvec(W_down, out["h_q8"], H, I, row_ids=ids)
    y_gpu = out["y"] if ids is None else out["y"][:, ids]
    assert oracle.within_tolerance(y_gpu, y_ref, T).all()


@pytest.mark.parametrize("H,I,nc", [(256, 256, 1), (512, 768, 2), (1024, 1280, 1), (768, 2048, 8), (3584, 512, 3)])
def test_ffn_small_stagewise_and_end_to_end(cuda_ready, variant, H, I, nc):
    mq = cuda_ready
    W_gu = synth.q4K_matrix(2 * I, H, seed=H + I, tag=synth.TAG_GU)
    W_down = synth.q4K_matrix(H, I, seed=H + I, tag=synth.TAG_DOWN)
    x = synth.activation(H, nc, seed=nc, tag=synth.TAG_X)
    out = _run(mq, W_gu, W_down, x, H, I)
    _stagewise(out, W_gu, W_down, x, H, I)
    out2 = _run(mq, W_gu, W_down, x, H, I, use_xq=True)
    for k in ("y", "h_q8", "gu", "h"):
        assert np.array_equal(out[k].view(np.uint8), out2[k].view(np.uint8)), k
    # end to end against the pure oracle chain
    y_ref, hq_ref = oracle.ffn(W_gu, W_down, x, H, I)
    wd = np.abs(dequant_rows(W_down, I))
    _, T = oracle.matvec(W_down, hq_ref, H, I)
    dh = np.abs(dequant_q8(out["h_q8"], I) - dequant_q8(hq_ref, I))      # [nc, I]
    widen = dh @ wd.T                                                    # [nc, H]
    assert np.all(np.abs(out["y"] - y_ref) <= 1e-3 * T + 1e-5 + widen * (1 + 1e-6))


def test_ffn_05b_layers_stagewise(cuda_ready, variant):
    mq = cuda_ready
    case = synth.FFN_05B
    for layer in (0, 11, 23):
        W_gu, W_down = synth.ffn_layer_weights(case, layer)
        x = synth.ffn_layer_input(case, layer)
        out = _run(mq, W_gu, W_down, x, case.H, case.I)
        _stagewise(out, W_gu, W_down, x, case.H, case.I)


@pytest.mark.parametrize("nc", [1, 2, 4, 8])
def test_ffn_7b_stagewise(cuda_ready, variant, nc):
    mq = cuda_ready
    case = synth.FFN_7B
    W_gu, W_down = synth.ffn_layer_weights(case, 0)
    x = synth.ffn_layer_input(case, 0, ncols=nc)
    out = _run(mq, W_gu, W_down, x, case.H, case.I)
    rng = np.random.default_rng(nc)
    gu_rows = None if nc == 1 else np.sort(rng.choice(2 * case.I, 512, replace=False))
    down_rows = None if nc == 1 else np.sort(rng.choice(case.H, 256, replace=False))
    _stagewise(out, W_gu, W_down, x, case.H, case.I, gu_rows=gu_rows, down_rows=down_rows)


def test_ffn_deterministic_aa(cuda_ready, variant):
    mq = cuda_ready
    case = synth.FFN_7B
    W_gu, W_down = synth.ffn_layer_weights(case, 0)
    x = synth.ffn_layer_input(case, 0)
    a = _run(mq, W_gu, W_down, x, case.H, case.I)
    b = _run(mq, W_gu, W_down, x, case.H, case.I)
    for k in ("y", "h_q8", "gu", "h"):
        assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k
