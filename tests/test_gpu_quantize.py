"""q8_0 quantization on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest

import oracle
from quantized_decode_matvec_gb300 import synth

pytestmark = pytest.mark.gpu


def _gpu_quant(mq, x_np):
    import torch
    x = torch.from_numpy(np.ascontiguousarray(x_np)).cuda()
    out = mq.quantize_q8_0(x)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("K,ncols", [(32, 1), (256, 1), (1024, 3), (3584, 1), (18944, 1), (18944, 8), (4864, 5)])
def test_bit_exact_random(cuda_ready, K, ncols):
    x = synth.activation(K, ncols, seed=K + ncols, tag=synth.TAG_X)
    got = _gpu_quant(cuda_ready, x)
    ref = oracle.quantize_q8_0(x)
    assert got.shape == ref.shape
    assert np.array_equal(got, ref)


def test_bit_exact_edge_values(cuda_ready):
    blocks = []
    z = np.zeros(32, np.float32)
    blocks.append(z.copy())                                        # all zero
    t = z.copy(); t[0] = 127; t[1:9] = [2.5, -2.5, 0.5, -0.5, 1.5, -1.5, 126.5, -126.5]
    blocks.append(t)                                               # exact ties
    blocks.append(np.full(32, 1e-30, np.float32))                  # scale underflows in f16
    blocks.append(np.linspace(-1e-6, 1e-6, 32).astype(np.float32))  # subnormal f16 scale
    blocks.append(np.linspace(-3e7, 5e7, 32).astype(np.float32))    # scale overflows f16
    blocks.append(-np.arange(32, dtype=np.float32))                # negative amax
    s = z.copy(); s[7] = -0.0; s[9] = 3.0                          # signed zero
    blocks.append(s)
    rng = np.random.default_rng(0)
    for _ in range(25):
        blocks.append((rng.standard_normal(32) * 10.0 ** rng.uniform(-8, 8)).astype(np.float32))
    x = np.concatenate(blocks).reshape(1, -1)
    got = _gpu_quant(cuda_ready, x)
    ref = oracle.quantize_q8_0(x)
    assert np.array_equal(got, ref)


def test_hunted_division_case(cuda_ready):
    # a block where x/d and x*(1/d) round to different codes: the GPU must divide
    from tests.test_oracle_q8_0 import _find_div_vs_recip_case
    amax, xv, q_div, q_rec = _find_div_vs_recip_case()
    blk = np.zeros((1, 32), np.float32)
    blk[0, 0] = amax
    blk[0, 1] = xv
    got = _gpu_quant(cuda_ready, blk)
    assert np.array_equal(got, oracle.quantize_q8_0(blk))
    assert int(got[0, 3].view(np.int8)) == q_div


def test_empty_is_noop(cuda_ready):
    import torch
    mq = cuda_ready
    x = torch.zeros((0, 64), dtype=torch.float32, device="cuda")
    out = mq.quantize_q8_0(x)
    torch.cuda.synchronize()
    assert out.shape == (0, 68)


def _near_tie_blocks(n_blocks: int, seed: int) -> np.ndarray:
    """Blocks whose values sit within a few ulps of (k + 1/2) * d, d = fp32(amax/127):
    the cases where an approximate quotient could round to the wrong code.  The
    first value of each block is +-amax, so every block keeps its own scale."""
    rng = np.random.default_rng(seed)
    amax = (rng.uniform(0.5, 2.0, n_blocks) * 10.0 ** rng.integers(-12, 13, n_blocks)).astype(np.float32)
    d = (amax / np.float32(127)).astype(np.float32)
    k = rng.integers(-127, 127, (n_blocks, 31)).astype(np.float32) + np.float32(0.5)
    c = (k * d[:, None]).astype(np.float32)
    # half within 3 ulps (the exact division decides), half within 400 ulps (mostly the fast path)
    span = np.where(rng.random(c.shape) < 0.5, 3, 400)
    off = np.rint((rng.random(c.shape) * 2 - 1) * span).astype(np.int32)
    nudged = (c.view(np.int32) + off).view(np.float32)
    x = np.where(np.abs(nudged) <= amax[:, None], nudged, c)
    x = np.where(np.abs(x) <= amax[:, None], x, np.float32(0))
    sign = np.where(rng.random(n_blocks) < 0.5, np.float32(-1), np.float32(1))
    return np.concatenate([(sign * amax)[:, None], x], axis=1).astype(np.float32)


@pytest.mark.parametrize("seed", [1, 2])
def test_near_tie_codes_bit_exact(cuda_ready, seed):
    """Values next to code boundaries, through the stand-alone quantizer and
    through the quantization fused into the matvec's staging (its q8_0 copy)."""
    import torch
    mq = cuda_ready
    x = _near_tie_blocks(4096, seed).reshape(1, -1)       # K = 131072
    ref = oracle.quantize_q8_0(x)
    assert np.array_equal(_gpu_quant(mq, x), ref)
    K = x.shape[1]
    W = torch.from_numpy(synth.q4K_matrix(8, K, seed=seed)).cuda()
    xq_out = torch.zeros((1, K // 32 * 34), dtype=torch.uint8, device="cuda")
    mq.matvec_q4K_q8_0(W, 8, K, x=torch.from_numpy(x).cuda(), xq_out=xq_out)
    torch.cuda.synchronize()
    assert np.array_equal(xq_out.cpu().numpy(), ref)
