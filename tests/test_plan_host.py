"""The launch planner on the host (mq_debug_plan_mv / mq_debug_plan_step): no GPU.

The planner decides, per call, which kernel family runs, how each row is
split into segments and lanes, the tile height and the shared-memory layout.
These tests check, for every shape and column count the library takes, that
a plan covers every unit of a row and every row of the matrix, fits the
device's shared memory and hands each warp a consistent share, and that the
persistent step kernel splits each phase's rows exactly as the per-matrix
kernels do, which is what makes the two step forms reduce in the same order.
The device descriptions are stated here (SM count, L2 bytes, opt-in shared
memory per block), so nothing depends on the machine the tests run on.
"""
import itertools

import pytest

# GB300 as the CUDA runtime reports it: 152 SMs, 126.5 MiB of L2, 227 KiB of
# opt-in shared memory per block; and a smaller device to exercise other limits
GB300 = dict(num_sms=152, l2_bytes=132644864, max_smem=232448)
SMALLER = dict(num_sms=100, l2_bytes=50 * 1024 * 1024, max_smem=166912)
Q4K_UNIT_BYTES = 72  # 128 weights of q4_K: half a 144-byte super-block


@pytest.fixture(scope="module")
def mq(mq_lib):
    return mq_lib


def check_plan(p, kind, rows, K, nc, I, dev):
    """Invariants every plan satisfies, whatever its kernel family."""
    assert p["variant"] in (0, 1)
    assert 1 <= p["grid"] and p["block"] % 32 == 0 and 128 <= p["block"] <= 1024
    assert 0 < p["smem"] <= dev["max_smem"]
    rows_done = p["grid"] * p["rows_per_cta"]
    assert rows_done >= (2 * I if kind == 2 else rows)
    if kind == 2:
        assert p["rows_per_cta"] % 64 == 0  # whole h blocks: 32 gate rows and their 32 up rows
    if p["variant"] == 0:  # register-streaming kernels: 64-weight chunks
        assert p["C"] == K // 64 and p["ksplit"] == 1
        return
    # bulk-copy ring kernels
    parts = p["ksplit"]
    assert parts >= 1
    if parts == 1:
        assert p["kpn"] == 0 and p["C"] == K // 128
    else:
        assert kind != 2 and p["kpn"] * parts * 256 == K and p["C"] == K // parts // 128
    L, S, nseg = p["L"], p["S"], p["nseg"]
    assert L in (4, 8, 16, 32) and 1 <= S <= L
    cu = 2 * p["C"] if p["hu"] else p["C"]  # units the split counts: half-units on half-unit lanes
    assert nseg * S >= cu and (nseg - 1) * S < cu  # every unit in exactly one segment, none empty
    assert p["block"] == 32 * (p["nwc"] + 1)  # consumers plus the bulk-copy warp
    assert 2 <= p["ns"] <= 8 and p["stage_bytes"] % 128 == 0
    assert 1 <= p["T"] and p["T"] * p["C"] * Q4K_UNIT_BYTES <= p["stage_bytes"]
    assert p["ns"] * p["stage_bytes"] < p["smem"]
    modes = p["hu"] + p["cmap"] + (1 if p["cgw"] and not p["hu"] else 0)
    assert modes <= 1
    if p["hu"]:
        assert nc in (4, 8)
        groups = nc // 4
    elif p["cgw"]:
        assert 3 <= nc <= 8
        groups = (nc + 1) // 2
    if p["hu"] or p["cgw"]:
        assert groups * p["cgw"] <= p["nwc"] <= 15
        assert p["cgu"] <= p["cgw"] and p["cgu"] % nseg == 0
        assert p["rg"] == (p["cgu"] // nseg) * (32 // L)
    elif p["cmap"]:
        assert nc >= 5 and p["rg"] == p["nwc"] // nseg
    else:
        assert p["nwc"] % nseg == 0 and p["rg"] == (p["nwc"] // nseg) * (32 // L)


SHAPES = [  # (kind, rows, K, I): matvec rows x K, down H x I, gate/up 2I x H
    (0, 1, 256, 0), (0, 7, 1024, 0), (0, 512, 1024, 0), (0, 4096, 4096, 0), (0, 4608, 3584, 0),
    (0, 3584, 3584, 0), (0, 4096, 14336, 0), (0, 4096, 18944, 0), (0, 333, 131072, 0),
    (1, 1024, 4864, 0), (1, 3584, 18944, 0), (1, 768, 2048, 0),
    (2, 9728, 1024, 4864), (2, 37888, 3584, 18944), (2, 4096, 768, 2048), (2, 512, 256, 256),
]


@pytest.mark.parametrize("dev", [GB300, SMALLER], ids=["gb300", "smaller"])
def test_every_plan_covers_its_rows_and_fits(mq, dev):
    planned = 0
    for (kind, rows, K, I), nc in itertools.product(SHAPES, range(1, 9)):
        if K * nc > mq.MQ_MAX_K_TIMES_NCOLS:
            continue
        try:
            p = mq.debug_plan_mv(kind, rows, K, nc, I, **dev)
        except mq.MQError as e:
            assert e.status == mq.MQ_ERR_UNSUPPORTED, (kind, rows, K, nc)
            continue
        check_plan(p, kind, rows, K, nc, I, dev)
        planned += 1
    assert planned >= 100


def test_7b_plans_are_the_ones_measured(mq):
    # the splits the profiles and measured tables describe, at the 7B shapes on GB300
    plan = lambda kind, rows, K, nc, I=0: mq.debug_plan_mv(kind, rows, K, nc, I, **GB300)
    gu1 = plan(2, 37888, 3584, 1, 18944)
    assert (gu1["variant"], gu1["grid"], gu1["block"], gu1["L"], gu1["nseg"]) == (1, 152, 480, 4, 7)
    assert gu1["rows_per_cta"] == 256  # 592 h blocks over 152 CTAs: at most 4 blocks of 64 rows
    dn1 = plan(1, 3584, 18944, 1)
    assert (dn1["block"], dn1["L"], dn1["nseg"], dn1["ksplit"]) == (512, 32, 5, 1)
    gu4 = plan(2, 37888, 3584, 4, 18944)
    assert (gu4["hu"], gu4["L"], gu4["nseg"], gu4["cgw"], gu4["cgu"]) == (1, 8, 7, 15, 14)
    dn4 = plan(1, 3584, 18944, 4)
    assert (dn4["hu"], dn4["ksplit"], dn4["nseg"], dn4["cgu"]) == (1, 1, 10, 10)  # 10 of 15 warps
    gu8 = plan(2, 37888, 3584, 8, 18944)
    assert (gu8["hu"], gu8["cgw"], gu8["cgu"], gu8["block"]) == (1, 7, 7, 480)  # two groups of 7 warps
    dn8 = plan(1, 3584, 18944, 8)  # eight staged columns of K = 18944 do not fit beside a ring
    assert (dn8["ksplit"], dn8["kpn"], dn8["C"], dn8["hu"], dn8["nseg"], dn8["cgu"]) == (2, 37, 74, 1, 5, 5)
    mv8 = plan(0, 4096, 18944, 8)
    assert mv8["ksplit"] == 2 and mv8["variant"] == 1


SPLIT_KEYS = ("C", "L", "S", "nseg", "rg", "cmap", "cgw", "cgu", "hu", "nwc")


def _step_shape(mq, n_layers, H, I, qkv_rows, o_rows, o_K, nc):
    return mq.StepShape(n_layers=n_layers, H=H, I=I, qkv_rows=qkv_rows, o_rows=o_rows, o_K=o_K, ncols=nc,
                        flags=mq.MQ_STEP_PERSISTENT, workspace=None)


STEPS = [  # (n_layers, H, I, qkv_rows, o_rows, o_K)
    (28, 3584, 18944, 4608, 3584, 3584),  # the 7B-class step
    (3, 512, 1024, 768, 512, 512),        # the small step of the GPU tests
    (24, 1024, 4864, 0, 0, 1024),         # the 0.5B FFN-only stack
    (2, 768, 2048, 1024, 768, 512),
]


@pytest.mark.parametrize("dev", [GB300, SMALLER], ids=["gb300", "smaller"])
@pytest.mark.parametrize("case", STEPS, ids=["7b", "small", "ffn05b", "odd"])
def test_persistent_phases_split_like_the_per_matrix_kernels(mq, case, dev):
    n_layers, H, I, qkv_rows, o_rows, o_K = case
    phases = [(0, qkv_rows, H, 0), (0, o_rows, o_K, 0), (2, 2 * I, H, I), (1, H, I, 0)]
    planned = 0
    for nc in range(1, 9):
        shape = _step_shape(mq, n_layers, H, I, qkv_rows, o_rows, o_K, nc)
        try:
            sp = mq.debug_plan_step(shape, **dev)
        except mq.MQError as e:
            # the kernel's shared memory cannot hold a phase's whole activation beside two stages
            assert e.status == mq.MQ_ERR_UNSUPPORTED
            continue
        planned += 1
        assert sp["grid"] == dev["num_sms"] and sp["block"] == 32 * (sp["nwc"] + 1) <= 512
        assert sp["smem"] <= dev["max_smem"] and 2 <= sp["ns"] <= 8
        assert sp["ws_bytes"] == mq.mq_step_workspace_bytes(shape)
        for name, (kind, rows, K, I_) in zip(mq.PHASES, phases):
            q = sp[name]
            if rows == 0:  # a projection left out
                assert q["variant"] == 0 and q["rows_per_cta"] == 0
                continue
            assert q["variant"] == 1 and q["stage_bytes"] == sp["stage_bytes"]
            assert q["nwc"] <= sp["nwc"]
            assert q["T"] * q["C"] * Q4K_UNIT_BYTES <= sp["stage_bytes"]
            assert sp["grid"] * q["rows_per_cta"] >= (2 * I if kind == 2 else rows)
            p = mq.debug_plan_mv(kind, rows, K, nc, I_, **dev)
            # the per-matrix kernel takes whole rows with the same split, so both
            # step forms sum every row's segments in the same order
            assert p["variant"] == 1 and p["ksplit"] == 1, (name, nc)
            assert {k: q[k] for k in SPLIT_KEYS} == {k: p[k] for k in SPLIT_KEYS}, (name, nc)
    assert planned >= 1
    if case[0] == 28 and dev is GB300:
        assert planned == 3  # the 7B step runs persistent at 1-3 columns


def test_plan_arguments_are_checked(mq):
    out = (mq.c_i64 * mq.MQ_PLAN_FIELDS)()
    call = lambda *a: mq.mq_debug_plan_mv(*a)
    g = (GB300["num_sms"], GB300["l2_bytes"], GB300["max_smem"])
    assert call(0, 512, 1024, 1, 0, *g, out, mq.MQ_PLAN_FIELDS) == mq.MQ_OK
    assert call(3, 512, 1024, 1, 0, *g, out, mq.MQ_PLAN_FIELDS) == mq.MQ_ERR_INVALID_ARG        # kind
    assert call(0, 512, 1024, 1, 0, *g, out, mq.MQ_PLAN_FIELDS - 1) == mq.MQ_ERR_INVALID_ARG    # n_out
    assert call(0, 512, 1024, 1, 0, *g, None, mq.MQ_PLAN_FIELDS) == mq.MQ_ERR_INVALID_ARG       # out
    assert call(0, 512, 1000, 1, 0, *g, out, mq.MQ_PLAN_FIELDS) == mq.MQ_ERR_SHAPE              # K % 256
    assert call(0, 512, 1024, 9, 0, *g, out, mq.MQ_PLAN_FIELDS) == mq.MQ_ERR_SHAPE              # ncols
    assert call(0, 0, 1024, 1, 0, *g, out, mq.MQ_PLAN_FIELDS) == mq.MQ_ERR_INVALID_ARG          # nothing to plan
    assert call(2, 1000, 1024, 1, 512, *g, out, mq.MQ_PLAN_FIELDS) == mq.MQ_ERR_SHAPE           # rows != 2I
    assert call(0, 512, 1024, 1, 0, 0, g[1], g[2], out, mq.MQ_PLAN_FIELDS) == mq.MQ_ERR_INVALID_ARG
    assert call(0, 512, 1024, 1, 0, g[0], g[1], 0, out, mq.MQ_PLAN_FIELDS) == mq.MQ_ERR_INVALID_ARG
    # a device with 8 KiB of shared memory per block: no plan
    assert call(0, 4096, 18944, 8, 0, g[0], g[1], 8192, out, mq.MQ_PLAN_FIELDS) == mq.MQ_ERR_UNSUPPORTED
    n = mq.MQ_STEP_PLAN_FIELDS + 4 * mq.MQ_PLAN_FIELDS
    sout = (mq.c_i64 * n)()
    shape = _step_shape(mq, 2, 512, 1024, 768, 512, 512, 1)
    assert mq.mq_debug_plan_step(shape, *g, sout, n) == mq.MQ_OK
    assert mq.mq_debug_plan_step(shape, *g, sout, n - 1) == mq.MQ_ERR_INVALID_ARG
    bad = _step_shape(mq, 2, 500, 1024, 768, 512, 512, 1)
    assert mq.mq_debug_plan_step(bad, *g, sout, n) == mq.MQ_ERR_SHAPE
