"""The seeded input generator: determinism and the workloads' distributions."""
import numpy as np

from quantized_decode_matvec_gb300 import synth
from tests.q4k_layout import unpack_fields


def test_deterministic_and_tagged():
    a = synth.q4K_matrix(16, 512, 0, synth.TAG_W)
    b = synth.q4K_matrix(16, 512, 0, synth.TAG_W)
    c = synth.q4K_matrix(16, 512, 0, synth.TAG_GU)
    d = synth.q4K_matrix(16, 512, 1, synth.TAG_W)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)
    assert a.shape == (16, 2 * 144) and a.dtype == np.uint8
    x1 = synth.activation(1024, 2, 0)
    x2 = synth.activation(1024, 2, 0)
    assert np.array_equal(x1, x2) and x1.dtype == np.float32 and x1.shape == (2, 1024)


def test_field_distributions():
    W = synth.q4K_matrix(2000, 1024, 0, synth.TAG_W)
    d, dmin, sc, m, q = unpack_fields(W.reshape(-1, 144))
    # scales/mins uniform in 0..63, quants uniform in 0..15
    for f, n in ((sc, 64), (m, 64), (q, 16)):
        counts = np.bincount(f.ravel(), minlength=n)
        assert counts.size == n
        exp = f.size / n
        assert np.all(np.abs(counts - exp) < 6 * np.sqrt(exp))
    # d = |N(0, 2e-3)|, dmin = |N(0, 1e-3)|: mean of |N(0, s)| = s * sqrt(2/pi)
    assert abs(d.mean() / (2e-3 * np.sqrt(2 / np.pi)) - 1) < 0.02
    assert abs(dmin.mean() / (1e-3 * np.sqrt(2 / np.pi)) - 1) < 0.02
    assert np.all(d >= 0) and np.all(dmin >= 0)
    # some d values are binary16 subnormals (< 2^-14)
    assert np.mean(d < 2.0 ** -14) > 0.005


def test_activation_outliers():
    x = synth.activation(1 << 20, 1, 3)
    big = np.abs(x) > 8
    assert 0.0006 < big.mean() < 0.0014
    assert abs(x[~big].std() - 1) < 0.01


def test_workload_byte_counts():
    assert synth.weight_bytes_step(synth.STEP_7B) == 3_670_474_752
    assert synth.weight_bytes_ffn(synth.FFN_05B) == 201_719_808
    assert synth.weight_bytes_ffn(synth.FFN_7B) == 114_573_312
