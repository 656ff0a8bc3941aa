"""The C ABI on the CPU: the library loads, exports every symbol mq.h declares,
and the host-side checks reject bad arguments before anything reaches CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "mq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(mq_[a-z0-9_A-Z]+)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_exports_every_declared_symbol(mq_lib):
    declared = _declared_functions()
    assert len(declared) >= 15
    lib = ctypes.CDLL(mq_lib.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(mq_lib.EXPORTS) == declared


def test_struct_sizes_match_header(mq_lib):
    # pointers are 8 bytes on both hosts; int32 fields follow them without padding
    assert ctypes.sizeof(mq_lib.MvDesc) == 5 * 8 + 4 * 4
    assert ctypes.sizeof(mq_lib.FfnDesc) == 8 * 8 + 4 * 4
    assert ctypes.sizeof(mq_lib.LayerDesc) == 2 * 56 + 80
    assert ctypes.sizeof(mq_lib.StepShape) == 8 * 4 + 8


def test_sizes(mq_lib):
    assert mq_lib.mq_q4K_row_bytes(3584) == 14 * 144
    assert mq_lib.mq_q4K_row_bytes(18944) == 74 * 144
    assert mq_lib.mq_q4K_row_bytes(100) == 0
    assert mq_lib.mq_q8_0_bytes(1024) == 32 * 34
    assert mq_lib.mq_q8_0_bytes(33) == 0
    assert mq_lib.mq_quant_block_elems(mq_lib.MQ_TYPE_Q4_K) == 256
    assert mq_lib.mq_quant_block_bytes(mq_lib.MQ_TYPE_Q4_K) == 144
    assert mq_lib.mq_quant_block_elems(mq_lib.MQ_TYPE_Q8_0) == 32
    assert mq_lib.mq_quant_block_bytes(mq_lib.MQ_TYPE_Q8_0) == 34
    assert mq_lib.mq_quant_block_bytes(99) == 0
    assert mq_lib.mq_quant_block_elems(mq_lib.MQ_TYPE_Q4_0) == 32
    assert mq_lib.mq_quant_block_bytes(mq_lib.MQ_TYPE_Q4_0) == 18
    assert mq_lib.mq_abi_version() == 3
    assert mq_lib.mq_status_string(0) == "ok"
    assert "shape" in mq_lib.mq_status_string(2)


def test_concat_rows_feasible_mirrors_preconditions(mq_lib):
    T = mq_lib.MQ_TYPE_Q4_K
    f = mq_lib.mq_concat_rows_feasible
    rb = 3584 // 256 * 144
    # gate + up of the 7B FFN: feasible
    assert f([T, T], [3584, 3584], [18944, 18944], [18944 * rb, 18944 * rb])
    # q|k|v
    assert f([T, T, T], [3584] * 3, [3584, 512, 512], [3584 * rb, 512 * rb, 512 * rb])
    assert not f([T], [3584], [10], [10 * rb])                            # fewer than two
    assert not f([T, mq_lib.MQ_TYPE_Q8_0], [3584, 3584], [1, 1], [rb, 3584 // 32 * 34])  # mixed types
    assert not f([T, T], [3584, 4096], [1, 1], [rb, 4096 // 256 * 144])   # different ne0
    assert not f([T, T], [300, 300], [1, 1], [0, 0])                      # ne0 not a block multiple
    assert not f([T, T], [3584, 3584], [2, 2], [2 * rb, 2 * rb + 1])      # byte length mismatch
    assert not f([99, 99], [256, 256], [1, 1], [144, 144])                # unknown type


def test_host_validation_rejects_before_launch(mq_lib):
    m = mq_lib
    # shapes
    assert m.mq_matvec_q4K_q8_0(0, 10, 100, 1) == m.MQ_ERR_SHAPE      # K % 256
    assert m.mq_matvec_q4K_q8_0(0, 10, 0, 1) == m.MQ_ERR_SHAPE        # K == 0
    assert m.mq_matvec_q4K_q8_0(0, -1, 256, 1) == m.MQ_ERR_SHAPE
    assert m.mq_matvec_q4K_q8_0(0, 10, 256, 9) == m.MQ_ERR_SHAPE      # ncols > 8
    assert m.mq_matvec_q4K_q8_0(0, 10, 256 * 1024, 1) == m.MQ_ERR_UNSUPPORTED
    assert m.mq_matvec_q4K_q8_0(0, 10, 32768, 8) == m.MQ_ERR_UNSUPPORTED  # K*ncols limit
    # empty work is a no-op even without a device
    assert m.mq_matvec_q4K_q8_0(0, 0, 256, 1) == m.MQ_OK
    assert m.mq_matvec_q4K_q8_0(0, 10, 256, 0) == m.MQ_OK
    assert m.mq_quantize_q8_0(0, 0, 0, 1) == m.MQ_OK
    assert m.mq_quantize_q8_0(0, 0, 64, 0) == m.MQ_OK
    # null / misaligned pointers
    assert m.mq_matvec_q4K_q8_0(0, 10, 256, 1) == m.MQ_ERR_INVALID_ARG
    assert m.mq_matvec_q4K_q8_0(0x1004, 10, 256, 1) == m.MQ_ERR_ALIGN
    assert m.mq_quantize_q8_0(0, 0x1000, 64, 1) == m.MQ_ERR_INVALID_ARG
    assert m.mq_quantize_q8_0(0x1002, 0x1000, 64, 1) == m.MQ_ERR_ALIGN
    assert m.mq_quantize_q8_0(0x1000, 0x1001, 64, 1) == m.MQ_ERR_ALIGN
    assert m.mq_quantize_q8_0(0x1000, 0x1000, 48, 1) == m.MQ_ERR_SHAPE
    for fn in (m.mq_matvec_q4_0_q8_0, m.mq_matvec_q8_0_q8_0):  # other weight types: same checks
        assert fn(0, 10, 100, 1) == m.MQ_ERR_SHAPE
        assert fn(0, 10, 256, 9) == m.MQ_ERR_SHAPE
        assert fn(0, 0, 256, 1) == m.MQ_OK
        assert fn(0, 10, 256, 1) == m.MQ_ERR_INVALID_ARG
        assert fn(0x1004, 10, 256, 1) == m.MQ_ERR_ALIGN
    assert m.mq_ffn_gu_silu_down(0, 3584, 100, 1) == m.MQ_ERR_SHAPE
    assert m.mq_ffn_gu_silu_down(0, 3584, 18944, 1) == m.MQ_ERR_INVALID_ARG
    assert m.mq_step(0, m.StepShape(0, 3584, 18944, 4608, 3584, 3584, 1, 0)) == m.MQ_OK   # no layers
    assert m.mq_step(0, m.StepShape(2, 3584, 18944, 4608, 3584, 3584, 1, 0)) == m.MQ_ERR_INVALID_ARG
    assert m.mq_step(0x1004, m.StepShape(2, 3584, 18944, 4608, 3584, 3584, 1, 0)) == m.MQ_ERR_ALIGN
    assert m.mq_step(0x1000, m.StepShape(2, 3584, 100, 4608, 3584, 3584, 1, 0)) == m.MQ_ERR_SHAPE
    assert m.mq_concat_rows(0, [0, 0], [1, 1], m.MQ_TYPE_Q4_K, 256) == m.MQ_ERR_INVALID_ARG
    assert m.mq_concat_rows(0x1000, [0x2000, 0x3000], [1, 1], m.MQ_TYPE_Q4_K, 100) == m.MQ_ERR_SHAPE


def test_check_descriptors_on_host(mq_lib):
    m = mq_lib
    good = m.MvDesc(0x10000, 0, 0x20002, 0, 0x30004, 64, 512, 2, 64)
    assert m.mq_check_mv_desc(good) == m.MQ_OK
    bad_w = m.MvDesc(0x10008, 0, 0x20002, 0, 0x30004, 64, 512, 2, 64)
    assert m.mq_check_mv_desc(bad_w) == m.MQ_ERR_ALIGN
    bad_ld = m.MvDesc(0x10000, 0, 0x20002, 0, 0x30004, 64, 512, 2, 63)
    assert m.mq_check_mv_desc(bad_ld) == m.MQ_ERR_SHAPE
    no_act = m.MvDesc(0x10000, 0, 0, 0, 0x30004, 64, 512, 1, 64)
    assert m.mq_check_mv_desc(no_act) == m.MQ_ERR_INVALID_ARG
    bad_x = m.MvDesc(0x10000, 0x20002, 0, 0, 0x30004, 64, 512, 1, 64)
    assert m.mq_check_mv_desc(bad_x) == m.MQ_ERR_ALIGN
    f = m.FfnDesc(0x10000, 0x20000, 0x30000, 0, 0x40002, 0, 0, 0x50000, 3584, 18944, 1, 3584)
    assert m.mq_check_ffn_desc(f) == m.MQ_OK
    f.h_q8 = 0x40001
    assert m.mq_check_ffn_desc(f) == m.MQ_ERR_ALIGN
    f.h_q8 = 0x40002
    f.I = 1000
    assert m.mq_check_ffn_desc(f) == m.MQ_ERR_SHAPE


def test_binding_raises_without_fallback(mq_lib):
    # the tensor-level helpers surface library errors; there is no CPU path to fall back to
    with pytest.raises(mq_lib.MQError):
        mq_lib._check(mq_lib.mq_matvec_q4K_q8_0(0, 10, 100, 1), "x")


def test_persistent_step_needs_workspace(mq_lib):
    m = mq_lib
    # checked before any device work: no workspace, misaligned workspace
    shape = m.StepShape(2, 3584, 18944, 4608, 3584, 3584, 1, m.MQ_STEP_PERSISTENT, None)
    assert m.mq_step(0x1000, shape) == m.MQ_ERR_INVALID_ARG
    shape.workspace = 0x2002
    assert m.mq_step(0x1000, shape) == m.MQ_ERR_ALIGN
    shape.workspace = 0x2008  # the h records are read 16 bytes at a time
    assert m.mq_step(0x1000, shape) == m.MQ_ERR_ALIGN


def test_step_workspace_bytes(mq_lib):
    m = mq_lib
    # fixed words (abort word, one phase flag per CTA), then per column
    # 40 records of 8 bytes per 128 elements of h
    shape = m.StepShape(28, 3584, 18944, 4608, 3584, 3584, 1, m.MQ_STEP_PERSISTENT, None)
    assert m.mq_step_workspace_bytes(shape) == 4352 + 18944 // 128 * 320
    shape.ncols = 8
    assert m.mq_step_workspace_bytes(shape) == 4352 + 8 * (18944 // 128) * 320
    n = ctypes.c_size_t(0)
    lib = m._lib
    assert lib.mq_step_workspace_bytes(None, ctypes.byref(n)) == m.MQ_ERR_INVALID_ARG
    assert lib.mq_step_workspace_bytes(ctypes.byref(shape), None) == m.MQ_ERR_INVALID_ARG
    shape.I = 1000  # not a multiple of 256
    assert lib.mq_step_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)) == m.MQ_ERR_SHAPE


def test_chained_step_workspace_bytes(mq_lib):
    m = mq_lib
    # a chained step adds the output records of q|k|v, o and down: 8 bytes per output and column
    base = 4352 + 18944 // 128 * 320
    shape = m.StepShape(28, 3584, 18944, 4608, 3584, 3584, 1, m.MQ_STEP_PERSISTENT | m.MQ_STEP_CHAINED, None)
    assert m.mq_step_workspace_bytes(shape) == base + 8 * (4608 + 3584 + 3584)
    shape.ncols = 2
    assert m.mq_step_workspace_bytes(shape) == 4352 + 2 * (18944 // 128) * 320 + 16 * (4608 + 3584 + 3584)
    # an FFN-only chain: only down's outputs
    shape = m.StepShape(24, 1024, 4864, 0, 0, 0, 1, m.MQ_STEP_PERSISTENT | m.MQ_STEP_CHAINED, None)
    assert m.mq_step_workspace_bytes(shape) == 4352 + 4864 // 128 * 320 + 8 * 1024


def test_step_shapes_on_the_host(mq_lib):
    m = mq_lib
    # a stack of FFN layers only (q|k|v and o left out) is a valid shape; o_K is then ignored
    shape = m.StepShape(24, 1024, 4864, 0, 0, 0, 1, 0, None)
    assert m.mq_step_workspace_bytes(shape) == 4352 + 4864 // 128 * 320
    # negative rows and unknown flags are refused before any device work
    shape.qkv_rows = -1
    assert m.mq_step(0x1000, shape) == m.MQ_ERR_SHAPE
    shape.qkv_rows = 0
    shape.flags = 64
    assert m.mq_step(0x1000, shape) == m.MQ_ERR_INVALID_ARG
    # a projection that is present still needs a valid K
    shape = m.StepShape(2, 1000, 4864, 512, 0, 0, 1, 0, None)
    assert m.mq_step(0x1000, shape) == m.MQ_ERR_SHAPE
    shape = m.StepShape(2, 1024, 4864, 0, 512, 1000, 1, 0, None)
    assert m.mq_step(0x1000, shape) == m.MQ_ERR_SHAPE
