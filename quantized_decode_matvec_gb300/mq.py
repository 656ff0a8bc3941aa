"""Thin ctypes binding of libmq (include/mq.h), same call names as the C ABI.

Argument marshalling only: every step of the compute path runs in the CUDA
kernels of libmq.so.  There is no CPU fallback: importing this module raises
if the in-tree library has not been built, and every compute call raises
``MQError`` on a non-zero status.

Raw calls (``mq_*``) take integer device addresses and a stream handle.
The tensor-level helpers below them (``quantize_q8_0``, ``matvec_q4K_q8_0``,
``ffn_gu_silu_down``, ``StepBuffers``) only compute pointers from torch
tensors, build the descriptor structs and upload them.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libmq.so is not built ({LIB_PATH}); run `python -c 'import __graft_entry__ as g; g.build()'`")

_lib = ctypes.CDLL(LIB_PATH)

c_i32 = ctypes.c_int32
c_i64 = ctypes.c_int64
c_u32 = ctypes.c_uint32
c_vp = ctypes.c_void_p

MQ_OK = 0
MQ_ERR_INVALID_ARG = 1
MQ_ERR_SHAPE = 2
MQ_ERR_ALIGN = 3
MQ_ERR_CUDA = 4
MQ_ERR_UNSUPPORTED = 5
MQ_ERR_NOT_INITIALIZED = 6
MQ_DEV_DESC_MISMATCH = 1
MQ_DEV_DESC_ALIGN = 2
MQ_DEV_TIMEOUT = 4
MQ_DEV_ALIAS = 8
MQ_VARIANT_AUTO = 0
MQ_VARIANT_FORCE_REGISTER = 1
MQ_FAULT_NONE = 0
MQ_FAULT_WITHHOLD_TILE = 1
MQ_FAULT_WITHHOLD_RECORDS = 2
MQ_FAULT_WITHHOLD_COUNT = 3
MQ_TYPE_Q4_K = 1
MQ_TYPE_Q8_0 = 2
MQ_TYPE_Q4_0 = 3
MQ_MAX_NCOLS = 8
MQ_MAX_K = 131072
MQ_MAX_K_TIMES_NCOLS = 163840
MQ_STEP_PDL = 1
MQ_STEP_PERSISTENT = 2
MQ_STEP_CHAINED = 4
MQ_STEP_WORKSPACE_BYTES = 4352
MQ_NOALLOC_HQ8_MAX_BYTES = 131072
MQ_MMQ_MAX_NCOLS = 64
MQ_PLAN_MATVEC = 0
MQ_PLAN_DOWN = 1
MQ_PLAN_GATE_UP = 2
MQ_PLAN_FIELDS = 20
MQ_STEP_PLAN_FIELDS = 8


class MvDesc(ctypes.Structure):
    _fields_ = [("W", c_vp), ("x", c_vp), ("xq", c_vp), ("xq_out", c_vp), ("y", c_vp),
                ("rows", c_i32), ("K", c_i32), ("ncols", c_i32), ("y_ld", c_i32)]


class FfnDesc(ctypes.Structure):
    _fields_ = [("W_gu", c_vp), ("W_down", c_vp), ("x", c_vp), ("xq", c_vp), ("h_q8", c_vp),
                ("gu_dbg", c_vp), ("h_dbg", c_vp), ("y", c_vp),
                ("H", c_i32), ("I", c_i32), ("ncols", c_i32), ("y_ld", c_i32)]


class LayerDesc(ctypes.Structure):
    _fields_ = [("qkv", MvDesc), ("o", MvDesc), ("ffn", FfnDesc)]


class StepShape(ctypes.Structure):
    _fields_ = [("n_layers", c_i32), ("H", c_i32), ("I", c_i32), ("qkv_rows", c_i32), ("o_rows", c_i32),
                ("o_K", c_i32), ("ncols", c_i32), ("flags", c_u32), ("workspace", c_vp)]


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("mq_status_string", ctypes.c_char_p, c_i32)
_sig("mq_abi_version", c_i32)
_sig("mq_last_cuda_error", c_i32)
_sig("mq_init", c_i32, c_i32)
_sig("mq_read_device_status", c_i32, ctypes.POINTER(c_u32), c_vp)
_sig("mq_q4K_row_bytes", ctypes.c_size_t, c_i64)
_sig("mq_q8_0_bytes", ctypes.c_size_t, c_i64)
_sig("mq_quant_block_elems", c_i32, c_i32)
_sig("mq_quant_block_bytes", c_i32, c_i32)
_sig("mq_concat_rows_feasible", c_i32, c_i32, ctypes.POINTER(c_i32), ctypes.POINTER(c_i64),
     ctypes.POINTER(c_i64), ctypes.POINTER(ctypes.c_uint64))
_sig("mq_concat_rows", c_i32, c_vp, ctypes.POINTER(c_vp), ctypes.POINTER(c_i64), c_i32, c_i32, c_i64, c_vp)
_sig("mq_quantize_q8_0", c_i32, c_vp, c_vp, c_i64, c_i32, c_vp)
_sig("mq_check_mv_desc", c_i32, ctypes.POINTER(MvDesc))
_sig("mq_matvec_q4K_q8_0", c_i32, c_vp, c_i32, c_i32, c_i32, c_vp)
_sig("mq_matvec_q4_0_q8_0", c_i32, c_vp, c_i32, c_i32, c_i32, c_vp)
_sig("mq_matvec_q8_0_q8_0", c_i32, c_vp, c_i32, c_i32, c_i32, c_vp)
_sig("mq_check_ffn_desc", c_i32, ctypes.POINTER(FfnDesc))
_sig("mq_ffn_gu_silu_down", c_i32, c_vp, c_i32, c_i32, c_i32, c_vp)
_sig("mq_ffn_gate_up", c_i32, c_vp, c_i32, c_i32, c_i32, c_vp)
_sig("mq_step", c_i32, c_vp, ctypes.POINTER(StepShape), c_vp)
_sig("mq_step_workspace_bytes", c_i32, ctypes.POINTER(StepShape), ctypes.POINTER(ctypes.c_size_t))
_sig("mq_ffn_gu_silu_down_noalloc", c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp)
_sig("mq_mmq_workspace_bytes", c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(ctypes.c_size_t))
_sig("mq_mmq_q4K_q8_0", c_i32, c_vp, c_i32, c_i32, c_i32, c_vp, ctypes.c_size_t, c_vp)
_sig("mq_dequant_q4K_f16", c_i32, c_vp, c_vp, c_i64, c_i64, c_vp)
_sig("mq_convert_f32_f16", c_i32, c_vp, c_vp, c_i64, c_vp)
_sig("mq_gemm_f16", c_i32, c_vp, c_vp, c_vp, c_i32, c_i32, c_i32, c_vp)
_sig("mq_debug_block_sums_q4K_q8_0", c_i32, c_vp, c_i32, c_i32, c_i32, c_vp, c_vp, c_vp)
_sig("mq_debug_set_variant", c_i32, c_i32)
_sig("mq_debug_set_fault", c_i32, c_i32)
_sig("mq_debug_plan_mv", c_i32, c_i32, c_i64, c_i32, c_i32, c_i32, c_i32, c_i64, c_i32, ctypes.POINTER(c_i64), c_i32)
_sig("mq_debug_plan_step", c_i32, ctypes.POINTER(StepShape), c_i32, c_i64, c_i32, ctypes.POINTER(c_i64), c_i32)

# the exported names, one per declaration in include/mq.h
EXPORTS = ["mq_status_string", "mq_abi_version", "mq_last_cuda_error", "mq_init", "mq_read_device_status",
           "mq_q4K_row_bytes", "mq_q8_0_bytes", "mq_quant_block_elems", "mq_quant_block_bytes",
           "mq_concat_rows_feasible", "mq_concat_rows", "mq_quantize_q8_0", "mq_check_mv_desc",
           "mq_matvec_q4K_q8_0", "mq_matvec_q4_0_q8_0", "mq_matvec_q8_0_q8_0", "mq_check_ffn_desc", "mq_ffn_gu_silu_down", "mq_ffn_gate_up", "mq_step", "mq_step_workspace_bytes",
           "mq_ffn_gu_silu_down_noalloc", "mq_dequant_q4K_f16", "mq_convert_f32_f16", "mq_gemm_f16",
           "mq_mmq_workspace_bytes", "mq_mmq_q4K_q8_0",
           "mq_debug_block_sums_q4K_q8_0", "mq_debug_set_variant", "mq_debug_set_fault", "mq_debug_plan_mv",
           "mq_debug_plan_step"]


class MQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {mq_status_string(status)} (status {status})"
        if status == MQ_ERR_CUDA:
            msg += f", cudaError {mq_last_cuda_error()}"
        super().__init__(msg)


def status_string(s: int) -> str:
    return _lib.mq_status_string(s).decode()


# ---- raw calls, same names as the C ABI -------------------------------------------------------------

def mq_status_string(s: int) -> str:
    return status_string(s)


def mq_abi_version() -> int:
    return _lib.mq_abi_version()


def mq_last_cuda_error() -> int:
    return _lib.mq_last_cuda_error()


def mq_init(device: int) -> int:
    return _lib.mq_init(device)


def mq_read_device_status(stream: int = 0) -> int:
    v = c_u32(0)
    _check(_lib.mq_read_device_status(ctypes.byref(v), c_vp(stream)), "mq_read_device_status")
    return v.value


def mq_q4K_row_bytes(K: int) -> int:
    return _lib.mq_q4K_row_bytes(K)


def mq_q8_0_bytes(K: int) -> int:
    return _lib.mq_q8_0_bytes(K)


def mq_quant_block_elems(t: int) -> int:
    return _lib.mq_quant_block_elems(t)


def mq_quant_block_bytes(t: int) -> int:
    return _lib.mq_quant_block_bytes(t)


def mq_concat_rows_feasible(ttypes: Sequence[int], ne0: Sequence[int], ne1: Sequence[int],
                            nbytes: Sequence[int]) -> bool:
    n = len(ttypes)
    if not (len(ne0) == len(ne1) == len(nbytes) == n):
        return False
    A = lambda ct, v: (ct * n)(*v)
    return bool(_lib.mq_concat_rows_feasible(n, A(c_i32, ttypes), A(c_i64, ne0), A(c_i64, ne1),
                                             A(ctypes.c_uint64, nbytes)))


def mq_concat_rows(dst: int, srcs: Sequence[int], rows: Sequence[int], ttype: int, ne0: int,
                   stream: int = 0) -> int:
    n = len(srcs)
    return _lib.mq_concat_rows(c_vp(dst), (c_vp * n)(*srcs), (c_i64 * n)(*rows), n, ttype, ne0, c_vp(stream))


def mq_quantize_q8_0(x: int, xq: int, K: int, ncols: int, stream: int = 0) -> int:
    return _lib.mq_quantize_q8_0(c_vp(x), c_vp(xq), K, ncols, c_vp(stream))


def mq_check_mv_desc(d: MvDesc) -> int:
    return _lib.mq_check_mv_desc(ctypes.byref(d))


def mq_matvec_q4K_q8_0(d_desc: int, rows: int, K: int, ncols: int, stream: int = 0) -> int:
    return _lib.mq_matvec_q4K_q8_0(c_vp(d_desc), rows, K, ncols, c_vp(stream))


def mq_matvec_q4_0_q8_0(d_desc: int, rows: int, K: int, ncols: int, stream: int = 0) -> int:
    return _lib.mq_matvec_q4_0_q8_0(c_vp(d_desc), rows, K, ncols, c_vp(stream))


def mq_matvec_q8_0_q8_0(d_desc: int, rows: int, K: int, ncols: int, stream: int = 0) -> int:
    return _lib.mq_matvec_q8_0_q8_0(c_vp(d_desc), rows, K, ncols, c_vp(stream))


def mq_check_ffn_desc(d: FfnDesc) -> int:
    return _lib.mq_check_ffn_desc(ctypes.byref(d))


def mq_ffn_gu_silu_down(d_desc: int, H: int, I: int, ncols: int, stream: int = 0) -> int:
    return _lib.mq_ffn_gu_silu_down(c_vp(d_desc), H, I, ncols, c_vp(stream))


def mq_ffn_gate_up(d_desc: int, H: int, I: int, ncols: int, stream: int = 0) -> int:
    return _lib.mq_ffn_gate_up(c_vp(d_desc), H, I, ncols, c_vp(stream))


def mq_step(d_layers: int, shape: StepShape, stream: int = 0) -> int:
    return _lib.mq_step(c_vp(d_layers), ctypes.byref(shape), c_vp(stream))


def mq_step_workspace_bytes(shape: StepShape) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.mq_step_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)), "mq_step_workspace_bytes")
    return int(n.value)


def mq_ffn_gu_silu_down_noalloc(W_gu: int, W_down: int, x: int, xq: int, y: int, H: int, I: int, ncols: int,
                                y_ld: int, stream: int = 0) -> int:
    return _lib.mq_ffn_gu_silu_down_noalloc(c_vp(W_gu), c_vp(W_down), c_vp(x), c_vp(xq), c_vp(y), H, I, ncols,
                                            y_ld, c_vp(stream))


def mq_mmq_workspace_bytes(rows: int, K: int, ncols: int) -> int:
    n = ctypes.c_size_t(0)
    _check(_lib.mq_mmq_workspace_bytes(rows, K, ncols, ctypes.byref(n)), "mq_mmq_workspace_bytes")
    return int(n.value)


def mq_mmq_q4K_q8_0(d_desc: int, rows: int, K: int, ncols: int, workspace: int, ws_bytes: int,
                    stream: int = 0) -> int:
    return _lib.mq_mmq_q4K_q8_0(c_vp(d_desc), rows, K, ncols, c_vp(workspace), ws_bytes, c_vp(stream))


def mq_dequant_q4K_f16(W: int, W16: int, rows: int, K: int, stream: int = 0) -> int:
    return _lib.mq_dequant_q4K_f16(c_vp(W), c_vp(W16), rows, K, c_vp(stream))


def mq_convert_f32_f16(x: int, y: int, n: int, stream: int = 0) -> int:
    return _lib.mq_convert_f32_f16(c_vp(x), c_vp(y), n, c_vp(stream))


def mq_gemm_f16(W16: int, X16: int, Y: int, R: int, K: int, T: int, stream: int = 0) -> int:
    return _lib.mq_gemm_f16(c_vp(W16), c_vp(X16), c_vp(Y), R, K, T, c_vp(stream))


def mq_debug_block_sums_q4K_q8_0(d_desc: int, rows: int, K: int, ncols: int, sumi: int, sumq: int,
                                 stream: int = 0) -> int:
    return _lib.mq_debug_block_sums_q4K_q8_0(c_vp(d_desc), rows, K, ncols, c_vp(sumi), c_vp(sumq), c_vp(stream))


def mq_debug_set_variant(policy: int) -> int:
    return _lib.mq_debug_set_variant(policy)


def mq_debug_set_fault(fault: int) -> int:
    return _lib.mq_debug_set_fault(fault)


# the planner's fields, in the order mq.h gives them
PLAN_FIELDS = ("variant", "grid", "block", "smem", "C", "L", "S", "nseg", "nwc", "rg", "T", "ns", "stage_bytes",
               "rows_per_cta", "cmap", "cgw", "cgu", "hu", "ksplit", "kpn")
STEP_PLAN_FIELDS = ("grid", "block", "smem", "nwc", "ns", "stage_bytes", "pf_tiles", "ws_bytes")
PHASES = ("qkv", "o", "gu", "down")


def mq_debug_plan_mv(kind: int, rows: int, K: int, ncols: int, I: int, num_sms: int, l2_bytes: int,
                     max_smem: int, out, n_out: int) -> int:
    return _lib.mq_debug_plan_mv(kind, rows, K, ncols, I, num_sms, l2_bytes, max_smem, out, n_out)


def mq_debug_plan_step(shape: StepShape, num_sms: int, l2_bytes: int, max_smem: int, out, n_out: int) -> int:
    return _lib.mq_debug_plan_step(ctypes.byref(shape), num_sms, l2_bytes, max_smem, out, n_out)


def debug_plan_mv(kind: int, rows: int, K: int, ncols: int, I: int = 0, *, num_sms: int, l2_bytes: int,
                  max_smem: int) -> dict:
    """The plan a q4_K projection call takes on the stated device (host only), as a dict."""
    out = (c_i64 * MQ_PLAN_FIELDS)()
    _check(mq_debug_plan_mv(kind, rows, K, ncols, I, num_sms, l2_bytes, max_smem, out, MQ_PLAN_FIELDS),
           "mq_debug_plan_mv")
    return dict(zip(PLAN_FIELDS, list(out)))


def debug_plan_step(shape: StepShape, *, num_sms: int, l2_bytes: int, max_smem: int) -> dict:
    """The persistent step's plan on the stated device (host only): the kernel's fields and one
    dict per phase under "qkv", "o", "gu", "down"."""
    n = MQ_STEP_PLAN_FIELDS + 4 * MQ_PLAN_FIELDS
    out = (c_i64 * n)()
    _check(mq_debug_plan_step(shape, num_sms, l2_bytes, max_smem, out, n), "mq_debug_plan_step")
    v = list(out)
    d = dict(zip(STEP_PLAN_FIELDS, v[:MQ_STEP_PLAN_FIELDS]))
    for i, ph in enumerate(PHASES):
        o = MQ_STEP_PLAN_FIELDS + i * MQ_PLAN_FIELDS
        d[ph] = dict(zip(PLAN_FIELDS, v[o:o + MQ_PLAN_FIELDS]))
    return d


def _check(st: int, where: str):
    if st != MQ_OK:
        raise MQError(st, where)


# ---- tensor-level marshalling (torch owns memory and streams) ------------------------------------------

def _torch():
    import torch
    return torch


def _ptr(t) -> int:
    return 0 if t is None else t.data_ptr()


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


_initialized = set()


def init(device: Optional[int] = None) -> None:
    """mq_init for a device (default: torch's current device), once."""
    torch = _torch()
    dev = torch.cuda.current_device() if device is None else int(device)
    if dev in _initialized:
        return
    torch.cuda.init()
    _check(mq_init(dev), "mq_init")
    _initialized.add(dev)


def upload_struct(s: ctypes.Structure, device) -> "torch.Tensor":
    """Copy a descriptor struct to a new device buffer (8-byte aligned)."""
    torch = _torch()
    raw = bytes(s) if not isinstance(s, (bytes, bytearray)) else s
    host = torch.frombuffer(bytearray(raw), dtype=torch.uint8)
    return host.to(device)


def quantize_q8_0(x, out=None, stream=None):
    """fp32 [ncols, K] cuda tensor -> uint8 [ncols, K/32*34] q8_0."""
    torch = _torch()
    x2 = x if x.dim() == 2 else x.reshape(1, -1)
    ncols, K = x2.shape
    if out is None:
        out = torch.empty((ncols, K // 32 * 34), dtype=torch.uint8, device=x.device)
    _check(mq_quantize_q8_0(_ptr(x2), _ptr(out), K, ncols, _stream(stream)), "mq_quantize_q8_0")
    return out


def mv_desc(W, rows: int, K: int, y, x=None, xq=None, xq_out=None, ncols: int = 1,
            y_ld: Optional[int] = None) -> MvDesc:
    return MvDesc(_ptr(W), _ptr(x), _ptr(xq), _ptr(xq_out), _ptr(y), rows, K, ncols,
                  rows if y_ld is None else y_ld)


def matvec_q4K_q8_0(W, rows: int, K: int, x=None, xq=None, y=None, xq_out=None, ncols: Optional[int] = None,
                    stream=None):
    """y [ncols, rows] fp32 = W . q8_0(x) (or W . xq).  Returns (y, desc_buffer)."""
    torch = _torch()
    act = x if x is not None else xq
    if ncols is None:
        ncols = act.shape[0] if act.dim() == 2 else 1
    if y is None:
        y = torch.empty((ncols, rows), dtype=torch.float32, device=W.device)
    d = mv_desc(W, rows, K, y, x=x, xq=xq, xq_out=xq_out, ncols=ncols, y_ld=y.shape[-1])
    _check(mq_check_mv_desc(d), "mq_check_mv_desc")
    dd = upload_struct(d, W.device)
    _check(mq_matvec_q4K_q8_0(_ptr(dd), rows, K, ncols, _stream(stream)), "mq_matvec_q4K_q8_0")
    return y, dd


def matvec_w(wtype: str, W, rows: int, K: int, x=None, xq=None, y=None, ncols: Optional[int] = None, stream=None):
    """y [ncols, rows] fp32 = W . q8_0(x) (or W . xq) for q4_0 (``wtype="q4_0"``) or q8_0
    (``"q8_0"``) weights.  Returns (y, desc_buffer)."""
    torch = _torch()
    act = x if x is not None else xq
    if ncols is None:
        ncols = act.shape[0] if act.dim() == 2 else 1
    if y is None:
        y = torch.empty((ncols, rows), dtype=torch.float32, device=W.device)
    d = mv_desc(W, rows, K, y, x=x, xq=xq, ncols=ncols, y_ld=y.shape[-1])
    _check(mq_check_mv_desc(d), "mq_check_mv_desc")
    dd = upload_struct(d, W.device)
    fn = {"q4_0": mq_matvec_q4_0_q8_0, "q8_0": mq_matvec_q8_0_q8_0}[wtype]
    _check(fn(_ptr(dd), rows, K, ncols, _stream(stream)), f"mq_matvec_{wtype}_q8_0")
    return y, dd


def block_sums(W, rows: int, K: int, x=None, xq=None, ncols: Optional[int] = None, stream=None):
    """Test export: (sumi int32 [ncols, rows, K/32], sumq int32 [ncols, K/32])."""
    torch = _torch()
    act = x if x is not None else xq
    if ncols is None:
        ncols = act.shape[0] if act.dim() == 2 else 1
    y = torch.empty((ncols, rows), dtype=torch.float32, device=W.device)
    d = mv_desc(W, rows, K, y, x=x, xq=xq, ncols=ncols)
    _check(mq_check_mv_desc(d), "mq_check_mv_desc")
    dd = upload_struct(d, W.device)
    sumi = torch.empty((ncols, rows, K // 32), dtype=torch.int32, device=W.device)
    sumq = torch.empty((ncols, K // 32), dtype=torch.int32, device=W.device)
    _check(mq_debug_block_sums_q4K_q8_0(_ptr(dd), rows, K, ncols, _ptr(sumi), _ptr(sumq), _stream(stream)),
           "mq_debug_block_sums_q4K_q8_0")
    return sumi, sumq


def ffn_desc(W_gu, W_down, H: int, I: int, h_q8, y, x=None, xq=None, gu_dbg=None, h_dbg=None, ncols: int = 1,
             y_ld: Optional[int] = None) -> FfnDesc:
    return FfnDesc(_ptr(W_gu), _ptr(W_down), _ptr(x), _ptr(xq), _ptr(h_q8), _ptr(gu_dbg), _ptr(h_dbg), _ptr(y),
                   H, I, ncols, H if y_ld is None else y_ld)


def ffn_gu_silu_down(W_gu, W_down, H: int, I: int, x=None, xq=None, debug: bool = False, stream=None):
    """Fused FFN.  Returns dict with y [ncols, H], h_q8 and (debug) gu, h, plus the descriptor buffer."""
    torch = _torch()
    act = x if x is not None else xq
    ncols = act.shape[0] if act.dim() == 2 else 1
    dev = W_gu.device
    out = {
        "y": torch.empty((ncols, H), dtype=torch.float32, device=dev),
        "h_q8": torch.empty((ncols, I // 32 * 34), dtype=torch.uint8, device=dev),
    }
    if debug:
        out["gu"] = torch.empty((ncols, 2 * I), dtype=torch.float32, device=dev)
        out["h"] = torch.empty((ncols, I), dtype=torch.float32, device=dev)
    d = ffn_desc(W_gu, W_down, H, I, out["h_q8"], out["y"], x=x, xq=xq, gu_dbg=out.get("gu"), h_dbg=out.get("h"),
                 ncols=ncols)
    _check(mq_check_ffn_desc(d), "mq_check_ffn_desc")
    out["desc"] = upload_struct(d, dev)
    _check(mq_ffn_gu_silu_down(_ptr(out["desc"]), H, I, ncols, _stream(stream)), "mq_ffn_gu_silu_down")
    return out


def ffn_gu_silu_down_noalloc(W_gu, W_down, H: int, I: int, x=None, xq=None, y=None, stream=None):
    """mq_ffn_gu_silu_down_noalloc: the fused FFN with the library's own fixed
    scratch instead of a caller-owned h_q8 and descriptor.  Returns y [ncols, H]
    (allocated here by torch unless given)."""
    torch = _torch()
    act = x if x is not None else xq
    ncols = act.shape[0] if act.dim() == 2 else 1
    if y is None:
        y = torch.empty((ncols, H), dtype=torch.float32, device=W_gu.device)
    _check(mq_ffn_gu_silu_down_noalloc(_ptr(W_gu), _ptr(W_down), _ptr(x), _ptr(xq), _ptr(y), H, I, ncols,
                                       y.shape[-1], _stream(stream)), "mq_ffn_gu_silu_down_noalloc")
    return y


def mmq_q4K_q8_0(W, rows: int, K: int, x=None, xq=None, y=None, xq_out=None, ncols: Optional[int] = None,
                 workspace=None, stream=None):
    """The matmul for more columns on the tensor cores: y [ncols, rows] fp32 = W . q8_0(x) (or W . xq).
    Returns (y, desc_buffer, workspace)."""
    torch = _torch()
    act = x if x is not None else xq
    if ncols is None:
        ncols = act.shape[0] if act.dim() == 2 else 1
    if y is None:
        y = torch.empty((ncols, rows), dtype=torch.float32, device=W.device)
    nbytes = mq_mmq_workspace_bytes(rows, K, ncols)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 128), dtype=torch.uint8, device=W.device)
    d = mv_desc(W, rows, K, y, x=x, xq=xq, xq_out=xq_out, ncols=ncols, y_ld=y.shape[-1])
    dd = upload_struct(d, W.device)
    _check(mq_mmq_q4K_q8_0(_ptr(dd), rows, K, ncols, _ptr(workspace), workspace.numel(), _stream(stream)),
           "mq_mmq_q4K_q8_0")
    return y, dd, workspace


def dequant_q4K_f16(W, rows: int, K: int, out=None, stream=None):
    """The resident f16 weight cache: uint8 q4_K [rows, K/256*144] -> f16 [rows, K]."""
    torch = _torch()
    if out is None:
        out = torch.empty((rows, K), dtype=torch.float16, device=W.device)
    _check(mq_dequant_q4K_f16(_ptr(W), _ptr(out), rows, K, _stream(stream)), "mq_dequant_q4K_f16")
    return out


def convert_f32_f16(x, out=None, stream=None):
    """fp32 tensor -> f16 tensor of the same shape (round to nearest-even)."""
    torch = _torch()
    if out is None:
        out = torch.empty(x.shape, dtype=torch.float16, device=x.device)
    _check(mq_convert_f32_f16(_ptr(x), _ptr(out), x.numel(), _stream(stream)), "mq_convert_f32_f16")
    return out


def gemm_f16(W16, X16, out=None, stream=None):
    """Prefill GEMM on the tensor cores: Y [T, R] fp32 = X16 [T, K] . W16 [R, K]^T."""
    torch = _torch()
    R, K = W16.shape
    T = X16.shape[0]
    if out is None:
        out = torch.empty((T, R), dtype=torch.float32, device=W16.device)
    _check(mq_gemm_f16(_ptr(W16), _ptr(X16), _ptr(out), R, K, T, _stream(stream)), "mq_gemm_f16")
    return out


class StepBuffers:
    """Device buffers and the descriptor table of one layer stack for mq_step.

    weights: per layer dict with 'qkv' (concatenated q|k|v rows), 'o', 'gu', 'down'
    (uint8 cuda tensors); a stack of FFN layers only (qkv_rows == o_rows == 0)
    needs only 'gu' and 'down'.  Inputs a/b/c and outputs are allocated here, one
    buffer per layer, so a captured graph reads fresh inputs from the same
    addresses on every replay.

    chained: build the descriptors of a decode chain (MQ_STEP_CHAINED): the o
    projection reads the q|k|v output (its first o_K values), the FFN reads the
    o output, and layer l+1's q|k|v reads layer l's FFN output; only layer 0's
    first input (a[0], or c[0] for an FFN-only stack) comes from the caller.
    """

    def __init__(self, weights: List[Dict[str, "torch.Tensor"]], H: int, I: int, qkv_rows: int, o_rows: int,
                 o_K: int, ncols: int = 1, device=None, debug: bool = False, chained: bool = False):
        torch = _torch()
        self.n_layers = len(weights)
        self.H, self.I, self.qkv_rows, self.o_rows, self.o_K, self.ncols = H, I, qkv_rows, o_rows, o_K, ncols
        self.chained = chained
        dev = device if device is not None else weights[0]["gu"].device
        self.device = dev
        n = self.n_layers
        self.weights = weights
        if chained and ncols > 1 and ((qkv_rows and o_rows and qkv_rows != o_K) or (o_rows and o_rows != H)
                                      or (qkv_rows and not o_rows and qkv_rows != H)):
            raise ValueError("a chain of ncols > 1 needs each producer's rows equal to its consumer's K")
        # inputs [layer, ncols, K]: views of one buffer, so that a step's inputs
        # arrive in one host-to-device copy (each view starts on a 16-byte
        # boundary: H and o_K are multiples of 256)
        na, nb = n * ncols * H, n * ncols * o_K
        self.inputs = torch.zeros(na + nb + na, dtype=torch.float32, device=dev)
        self.a = self.inputs[:na].view(n, ncols, H)
        self.b = self.inputs[na:na + nb].view(n, ncols, o_K)
        self.c = self.inputs[na + nb:].view(n, ncols, H)
        # outputs: views of one buffer too (one device-to-host copy)
        nq, no = n * ncols * qkv_rows, n * ncols * o_rows
        self.outputs = torch.zeros(nq + no + n * ncols * H, dtype=torch.float32, device=dev)
        self.y_qkv = self.outputs[:nq].view(n, ncols, qkv_rows)
        self.y_o = self.outputs[nq:nq + no].view(n, ncols, o_rows)
        self.y_ffn = self.outputs[nq + no:].view(n, ncols, H)
        self.h_q8 = torch.zeros((n, ncols, I // 32 * 34), dtype=torch.uint8, device=dev)
        self.debug = debug
        if debug:
            self.xq_a = torch.zeros((n, ncols, H // 32 * 34), dtype=torch.uint8, device=dev)
            self.xq_b = torch.zeros((n, ncols, o_K // 32 * 34), dtype=torch.uint8, device=dev)
        table = (LayerDesc * n)()
        prev = None  # the fp32 output the next phase of a chain reads
        for l, w in enumerate(weights):
            if qkv_rows:
                xa = prev if (chained and prev is not None) else self.a[l]
                table[l].qkv = mv_desc(w["qkv"], qkv_rows, H, self.y_qkv[l], x=xa,
                                       xq_out=self.xq_a[l] if debug else None, ncols=ncols, y_ld=qkv_rows)
                prev = self.y_qkv[l]
            if o_rows:
                xb = prev if (chained and prev is not None) else self.b[l]
                table[l].o = mv_desc(w["o"], o_rows, o_K, self.y_o[l], x=xb,
                                     xq_out=self.xq_b[l] if debug else None, ncols=ncols, y_ld=o_rows)
                prev = self.y_o[l]
            xc = prev if (chained and prev is not None) else self.c[l]
            table[l].ffn = ffn_desc(w["gu"], w["down"], H, I, self.h_q8[l], self.y_ffn[l], x=xc,
                                    ncols=ncols, y_ld=H)
            prev = self.y_ffn[l]
            for rows, part in ((qkv_rows, table[l].qkv), (o_rows, table[l].o)):
                if rows:
                    _check(mq_check_mv_desc(part), "mq_check_mv_desc")
            _check(mq_check_ffn_desc(table[l].ffn), "mq_check_ffn_desc")
        self.table_host = table
        self.table = upload_struct(bytes(table), dev)
        # dependency words and records of the persistent step (zeroed by mq_step itself)
        nbytes = mq_step_workspace_bytes(StepShape(n, H, I, qkv_rows, o_rows, o_K, ncols,
                                                   MQ_STEP_CHAINED if chained else 0, None))
        self.workspace = torch.zeros(nbytes, dtype=torch.uint8, device=dev)

    def shape(self, flags: int = 0) -> StepShape:
        if self.chained:
            flags |= MQ_STEP_CHAINED
        return StepShape(self.n_layers, self.H, self.I, self.qkv_rows, self.o_rows, self.o_K, self.ncols, flags,
                         _ptr(self.workspace))

    def step(self, stream=None, flags: int = 0) -> None:
        _check(mq_step(_ptr(self.table), self.shape(flags), _stream(stream)), "mq_step")
