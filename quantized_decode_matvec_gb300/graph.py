"""Graph-resident decode step: capture mq_step once, replay it per token.

"Part 4 . Lecture 08 -- Graph-Resident Decode": capture the whole decode step
as one CUDA graph and replay it (Overview, section 1); everything that varies
per replay lives in device buffers the graph reads (section 2); lazy state is
pre-warmed before capture and a failed capture degrades to eager launches
with a log line instead of failing the run (section 3).

Here the per-replay state is the input of every layer, fed through the fixed
device buffers of ``StepBuffers`` (copied there from pinned host memory
before each replay); the descriptors and the grid sizes are fixed at capture.
"""
from __future__ import annotations

import contextlib
import logging
from typing import Callable, Optional

import torch

from . import mq

log = logging.getLogger("quantized_decode_matvec_gb300.graph")


class StepGraph:
    """Captured mq_step over a StepBuffers, with eager fallback.

    ``io`` (optional): a pair of pinned host tensors shaped like
    ``bufs.inputs`` and ``bufs.outputs``; the step then copies the inputs in
    and the outputs out as part of the same graph (one launch per step from
    host buffers to host buffers).  ``capture_hook`` (test-only) runs inside
    the capture window, so a test can plant a capture-illegal host operation
    and check the fallback.
    """

    def __init__(self, bufs: "mq.StepBuffers", flags: int = 0, use_graph: bool = True,
                 capture_hook: Optional[Callable[[], None]] = None, warmup: int = 1,
                 stream: Optional[torch.cuda.Stream] = None, io: Optional[tuple] = None):
        self.bufs = bufs
        self.flags = flags
        self.io = io
        self.stream = stream if stream is not None else torch.cuda.Stream(device=bufs.device)
        self.graph: Optional[torch.cuda.CUDAGraph] = None
        self.captured = False
        self.capture_error: Optional[str] = None
        mq.init(bufs.device.index if bufs.device.index is not None else torch.cuda.current_device())
        # warm-up outside the capture (pre-warms anything lazy on the torch side too)
        with torch.cuda.stream(self.stream):
            for _ in range(warmup):
                bufs.step(self.stream, flags)
        self.stream.synchronize()
        if use_graph:
            self._capture(capture_hook)

    def _capture(self, hook):
        # keep the captured cudaGraph_t (where this torch can) so that its nodes can be counted
        try:
            g = torch.cuda.CUDAGraph(keep_graph=True)
            self._kept = True
        except TypeError:
            g = torch.cuda.CUDAGraph()
            self._kept = False
        try:
            with torch.cuda.graph(g, stream=self.stream):
                if hook is not None:
                    hook()
                self._step()
        except Exception as e:  # capture failure: fall back to eager, keep running
            self.capture_error = f"{type(e).__name__}: {e}"
            log.warning("mq_step capture failed, running eagerly: %s", self.capture_error)
            self.graph = None
            self.captured = False
            try:
                torch.cuda.synchronize()
            except Exception:
                pass
            return
        if self._kept:
            try:
                self._nodes = _count_kernel_nodes(g.raw_cuda_graph())
                g.instantiate()  # else the first replay instantiates it
            except Exception as e:
                log.info("graph node count unavailable: %s", e)
        self.graph = g
        self.captured = True

    def run(self) -> None:
        """One decode step on self.stream: graph replay, or eager launches after a failed capture.

        CUDAGraph.replay() launches on torch's current stream, so make self.stream current.
        """
        with torch.cuda.stream(self.stream):
            if self.captured:
                self.graph.replay()
            else:
                self._step()

    def _step(self) -> None:
        # on self.stream (current): inputs in, the step, outputs out
        if self.io is not None:
            self.bufs.inputs.copy_(self.io[0], non_blocking=True)
        self.bufs.step(self.stream, self.flags)
        if self.io is not None:
            self.io[1].copy_(self.bufs.outputs, non_blocking=True)

    def node_count(self) -> Optional[int]:
        """Kernel nodes in the captured graph (None if not captured or not queryable)."""
        if not self.captured:
            return None
        return getattr(self, "_nodes", None)


def _count_kernel_nodes(raw: int) -> Optional[int]:
    """Kernel nodes of a cudaGraph_t (the driver's CUgraph), through the driver API;
    None if the driver library or the call is not available."""
    try:
        import ctypes
        cu = ctypes.CDLL("libcuda.so.1")
        n = ctypes.c_size_t(0)
        if cu.cuGraphGetNodes(ctypes.c_void_p(raw), None, ctypes.byref(n)) != 0:
            return None
        nodes = (ctypes.c_void_p * max(n.value, 1))()
        if cu.cuGraphGetNodes(ctypes.c_void_p(raw), nodes, ctypes.byref(n)) != 0:
            return None
        kinds = ctypes.c_int(0)
        count = 0
        for i in range(n.value):
            if cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(kinds)) != 0:
                return None
            count += kinds.value == 0  # CU_GRAPH_NODE_TYPE_KERNEL
        return count
    except Exception:
        return None


class PinnedFeeder:
    """Pinned host staging for the per-replay inputs of a StepBuffers.

    ``load(a, b, c)`` copies host arrays into the pinned buffers; ``push(stream)``
    enqueues the host-to-device copies into the fixed device input buffers.
    The pinned buffers are allocated once (size of all layers' inputs).
    """

    def __init__(self, bufs: "mq.StepBuffers"):
        self.bufs = bufs
        # one pinned buffer laid out like the device inputs (a, b, c views)
        self.inputs = torch.empty(bufs.inputs.shape, dtype=torch.float32, pin_memory=True)
        na, nb = bufs.a.numel(), bufs.b.numel()
        self.a = self.inputs[:na].view(bufs.a.shape)
        self.b = self.inputs[na:na + nb].view(bufs.b.shape)
        self.c = self.inputs[na + nb:].view(bufs.c.shape)

    @property
    def h2d_bytes(self) -> int:
        return self.inputs.numel() * 4

    def load(self, a, b, c) -> None:
        self.a.copy_(torch.as_tensor(a).reshape(self.a.shape))
        self.b.copy_(torch.as_tensor(b).reshape(self.b.shape))
        self.c.copy_(torch.as_tensor(c).reshape(self.c.shape))

    def push(self, stream) -> None:
        with torch.cuda.stream(stream):
            self.bufs.inputs.copy_(self.inputs, non_blocking=True)  # one host-to-device copy


class PinnedReadback:
    """Device-to-host readback through a self-held pinned staging buffer.

    "07 · R3 — small-model per-token overhead", A2 (the pinned readback): a
    read copies the device bytes into a page-locked buffer that this object
    keeps (one DMA, no bounce through the driver's own staging) and then into
    the caller's host tensor with an ordinary host copy.  The buffer is
    allocated on first use and replaced by a larger one when a read needs more
    than it holds; it is never smaller than ``min_bytes`` (4 MiB), so that
    small changes in the read size do not reallocate it.  When page-locked
    memory cannot be had, the read copies straight into the caller's pageable
    tensor and a warning is logged once per process; the next read tries the
    allocation again.

    ``pinned=False`` always takes the pageable path (an A/B switch).
    ``alloc`` (test hook) replaces the allocator: ``alloc(nbytes)`` returns a
    1-D uint8 host tensor or raises, which lets a host-only test plant an
    allocation failure.
    """

    MIN_BYTES = 4 * 1024 * 1024
    _warned = False  # one warning per process

    def __init__(self, pinned: bool = True, min_bytes: int = MIN_BYTES,
                 alloc: Optional[Callable[[int], torch.Tensor]] = None):
        self.pinned = pinned
        self.min_bytes = int(min_bytes)
        self._alloc = alloc if alloc is not None else self._alloc_pinned
        self._buf: Optional[torch.Tensor] = None
        self.allocations = 0  # buffers allocated (the first one and each growth)
        self.fallbacks = 0    # reads that took the pageable path after a failed allocation

    @staticmethod
    def _alloc_pinned(nbytes: int) -> torch.Tensor:
        return torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)

    @property
    def capacity(self) -> int:
        """Bytes of the pinned buffer held now (0 before the first read or after a failure)."""
        return 0 if self._buf is None else self._buf.numel()

    def _staging(self, nbytes: int) -> Optional[torch.Tensor]:
        if self._buf is not None and self._buf.numel() >= nbytes:
            return self._buf
        self._buf = None  # release the smaller buffer before asking for the larger one
        need = max(nbytes, self.min_bytes)
        try:
            buf = self._alloc(need)
        except (RuntimeError, MemoryError) as e:
            if not PinnedReadback._warned:
                PinnedReadback._warned = True
                log.warning("pinned readback buffer of %d bytes not allocated (%s); "
                            "reading through pageable memory", need, e)
            return None
        if buf.dtype != torch.uint8 or buf.dim() != 1 or buf.numel() < need:
            raise ValueError("readback allocator returned a buffer of the wrong type or size")
        self._buf = buf
        self.allocations += 1
        return buf

    def read_into(self, dst: torch.Tensor, src: torch.Tensor, stream=None) -> torch.Tensor:
        """Copy ``src`` (a contiguous tensor, normally on the GPU) into the contiguous host
        tensor ``dst`` of the same dtype and number of elements; returns ``dst``.

        The device-to-host copy runs on ``stream`` (torch's current stream if None) and is
        complete when this returns.
        """
        if dst.device.type != "cpu" or not dst.is_contiguous() or not src.is_contiguous():
            raise ValueError("read_into needs a contiguous host dst and a contiguous src")
        if dst.dtype != src.dtype or dst.numel() != src.numel():
            raise ValueError("dst and src differ in dtype or element count")
        nbytes = src.numel() * src.element_size()
        if nbytes == 0:
            return dst
        st = self._staging(nbytes) if self.pinned else None
        on_gpu = src.device.type == "cuda"
        ctx = torch.cuda.stream(stream) if (on_gpu and stream is not None) else contextlib.nullcontext()
        with ctx:
            if st is None:
                if self.pinned:
                    self.fallbacks += 1
                dst.copy_(src)  # pageable: the copy blocks until the bytes are in dst
                return dst
            stage = st[:nbytes]
            stage.copy_(src.reshape(-1).view(torch.uint8), non_blocking=on_gpu)
            if on_gpu:
                torch.cuda.current_stream().synchronize()
        dst.reshape(-1).view(torch.uint8).copy_(stage)  # host to host
        return dst

    def read(self, src: torch.Tensor, stream=None) -> torch.Tensor:
        """A new host tensor with the contents of ``src`` (same dtype and shape)."""
        return self.read_into(torch.empty(src.shape, dtype=src.dtype), src.contiguous(), stream)

