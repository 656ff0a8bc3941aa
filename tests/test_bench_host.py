"""Host-side parts of bench.py: the oracle's all-threads arm (static row
partition) gives the same bytes as the oracle's own single-threaded calls, so
the CPU baseline times the same computation on more threads."""
import numpy as np

import bench
import oracle
from quantized_decode_matvec_gb300 import synth


def test_host_cores_positive():
    assert bench.host_cores() >= 1


def test_threaded_matvec_equals_oracle():
    W = synth.q4K_matrix(97, 512, seed=50)
    x = synth.activation(512, 2, seed=51)
    xq = oracle.quantize_q8_0(x)
    ref = oracle.matvec(W, xq, 97, 512)[0]
    for t in (1, 3, 8):
        arm = bench.OracleArm(t)
        got = arm.matvec(W, xq, 97, 512)
        arm.close()
        assert np.array_equal(got.view(np.uint64), ref.view(np.uint64)), t


def test_threaded_matvec_w_equals_oracle():
    W = synth.wq_matrix("q4_0", 40, 256, seed=52)
    xq = oracle.quantize_q8_0(synth.activation(256, 1, seed=53))
    ref = oracle.matvec_w("q4_0", W, xq, 40, 256)[0]
    arm = bench.OracleArm(4)
    got = arm.matvec_w("q4_0", W, xq, 40, 256)
    arm.close()
    assert np.array_equal(got, ref)


def test_threaded_ffn_equals_oracle_chain():
    H, I = 256, 512
    W_gu = synth.q4K_matrix(2 * I, H, seed=54, tag=synth.TAG_GU)
    W_down = synth.q4K_matrix(H, I, seed=54, tag=synth.TAG_DOWN)
    x = synth.activation(H, 3, seed=55)
    ref = oracle.ffn(W_gu, W_down, x, H, I)[0]
    arm = bench.OracleArm(4)
    got = arm.ffn(W_gu, W_down, x, H, I)
    arm.close()
    assert np.array_equal(got, ref)


def test_oracle_step_runs_every_layer():
    case = synth.StepCase("tiny", 2, 256, 256, 256, 256, 1, 3)
    weights = bench.host_step_weights(case)
    inputs = [synth.step_layer_inputs(case, l, 0) for l in range(case.n_layers)]
    arm = bench.OracleArm(2)
    assert arm.step(case, weights, inputs) > 0.0
    arm.close()
