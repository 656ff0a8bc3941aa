"""Host-side logic of the pinned readback (graph.PinnedReadback).

"07 · R3 — small-model per-token overhead", A2: a self-held page-locked
staging buffer, at least 4 MiB, grown when a read needs more; a failed
page-locked allocation falls back to a pageable copy with one warning.  The
allocator is replaced by a test hook here (plain host tensors, or one that
raises), so these run without a GPU; the round trip from device memory is in
tests/test_gpu_step.py.
"""
import logging

import pytest
import torch

from quantized_decode_matvec_gb300.graph import PinnedReadback

MIB = 1024 * 1024


class FakeAlloc:
    """Pageable stand-in for the page-locked allocator; records the sizes asked for."""

    def __init__(self, fail=False):
        self.sizes = []
        self.fail = fail

    def __call__(self, nbytes):
        self.sizes.append(nbytes)
        if self.fail:
            raise RuntimeError("simulated page-locked allocation failure")
        return torch.empty(nbytes, dtype=torch.uint8)


@pytest.fixture(autouse=True)
def fresh_warning():
    PinnedReadback._warned = False
    yield
    PinnedReadback._warned = False


def _data(n, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(n, generator=g)


def test_grows_past_the_initial_buffer_and_keeps_it():
    a = FakeAlloc()
    r = PinnedReadback(alloc=a)
    assert r.capacity == 0
    small = _data(256, 1)                      # 1 KiB: the first buffer is the 4 MiB floor
    assert torch.equal(r.read(small), small)
    assert a.sizes == [4 * MIB] and r.capacity == 4 * MIB
    big = _data(1_400_000, 2)                  # 5.6 MB, larger than the first buffer
    out = r.read(big)
    assert torch.equal(out, big)
    assert a.sizes == [4 * MIB, 5_600_000] and r.capacity == 5_600_000
    again = _data(300, 3)                      # smaller again: the larger buffer is kept
    assert torch.equal(r.read(again), again)
    assert len(a.sizes) == 2 and r.allocations == 2 and r.fallbacks == 0


def test_exact_bytes_for_other_dtypes_and_shapes():
    r = PinnedReadback(alloc=FakeAlloc(), min_bytes=64)
    for t in (torch.arange(12, dtype=torch.int64).reshape(3, 4),
              torch.tensor([[1.5, -0.0], [float("inf"), float("nan")]], dtype=torch.float32),
              torch.arange(255, dtype=torch.uint8)):
        out = r.read(t)
        assert out.shape == t.shape and out.dtype == t.dtype
        assert torch.equal(out.reshape(-1).view(torch.uint8), t.reshape(-1).view(torch.uint8))


def test_failed_allocation_falls_back_to_pageable_and_warns_once(caplog):
    a = FakeAlloc(fail=True)
    r1, r2 = PinnedReadback(alloc=a), PinnedReadback(alloc=a)
    x = _data(1000, 4)
    with caplog.at_level(logging.WARNING, logger="quantized_decode_matvec_gb300.graph"):
        assert torch.equal(r1.read(x), x)
        assert torch.equal(r1.read(x), x)
        assert torch.equal(r2.read(x), x)
    warnings = [rec for rec in caplog.records if "pinned readback" in rec.getMessage()]
    assert len(warnings) == 1                  # once per process, not per read or per object
    assert r1.fallbacks == 2 and r2.fallbacks == 1 and r1.capacity == 0
    assert len(a.sizes) == 3                   # every read asked again
    a.fail = False                             # the allocation works again: the next read is staged
    assert torch.equal(r1.read(x), x)
    assert r1.capacity == 4 * MIB and r1.fallbacks == 2


def test_pageable_switch_never_allocates():
    a = FakeAlloc()
    r = PinnedReadback(pinned=False, alloc=a)
    x = _data(5000, 5)
    assert torch.equal(r.read(x), x)
    assert a.sizes == [] and r.capacity == 0 and r.fallbacks == 0


def test_empty_read_allocates_nothing():
    a = FakeAlloc()
    r = PinnedReadback(alloc=a)
    out = r.read(torch.empty(0, 7))
    assert out.shape == (0, 7) and a.sizes == []


def test_bad_arguments_are_refused():
    r = PinnedReadback(alloc=FakeAlloc())
    x = torch.zeros(8)
    with pytest.raises(ValueError):
        r.read_into(torch.zeros(8, dtype=torch.float64), x)       # dtype differs
    with pytest.raises(ValueError):
        r.read_into(torch.zeros(9), x)                             # size differs
    with pytest.raises(ValueError):
        r.read_into(torch.zeros(16)[::2], x)                       # dst not contiguous
    bad = PinnedReadback(alloc=lambda n: torch.empty(n // 2, dtype=torch.uint8))
    with pytest.raises(ValueError):
        bad.read(x)                                                # allocator returned too little


def test_default_allocator_without_a_gpu_takes_the_pageable_path():
    if torch.cuda.is_available():
        pytest.skip("page-locked memory is available here")
    r = PinnedReadback()
    x = _data(100, 6)
    assert torch.equal(r.read(x), x)
    assert r.fallbacks == 1 and r.capacity == 0
