"""Python binding of libqz: quantize tensors on a GB300 to INT8 / FP8 E4M3 / FP8 E5M2 /
MXFP4 / NVFP4, dequantize them, and measure the quantization error.

The functions ``qz_*`` mirror the C ABI of ``include/qz.h`` one to one (same names, same
arguments, device pointers as integers).  ``quantize`` / ``dequantize`` / ``error_stats`` /
``amax`` marshal torch tensors into those calls.  Every step of the computation runs in
the CUDA kernels of ``libqz.so``; there is no other code path, and importing the binding
fails if the library has not been built (``__graft_entry__.build()``).

Formats and semantics: blog post "浅谈低精度浮点数" (A brief talk on low-precision floats),
sections "FP8" and "FP4 / MXFP4 / NVFP4"; see include/qz.h for the exact rules.
"""
from __future__ import annotations

import ctypes as C
import os
import struct
from dataclasses import dataclass

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqz.so")

# ---- enums (values of include/qz.h) ----
QZ_OK, QZ_ERR_NULL, QZ_ERR_ENUM, QZ_ERR_SHAPE, QZ_ERR_ALIGN = 0, 1, 2, 3, 4
QZ_ERR_UNSUPPORTED, QZ_ERR_CUDA, QZ_ERR_WORKSPACE = 5, 6, 7
QZ_INT8, QZ_FP8_E4M3, QZ_FP8_E5M2, QZ_MXFP4, QZ_NVFP4, QZ_INT4 = 1, 2, 3, 4, 5, 6
QZ_BF16, QZ_F32 = 1, 2
QZ_GRAN_TENSOR, QZ_GRAN_ROW, QZ_GRAN_BLOCK, QZ_GRAN_UNIT = 1, 2, 3, 4
QZ_ROUND_RNE = 0
QZ_SCALE_UP, QZ_SCALE_NEAREST = 0, 1
QZ_FLAG_NONFINITE_INPUT, QZ_FLAG_BAD_AMAX, QZ_FLAG_PIPELINE_TIMEOUT = 0x1, 0x2, 0x4

FORMATS = {"int8": QZ_INT8, "e4m3": QZ_FP8_E4M3, "e5m2": QZ_FP8_E5M2,
           "mxfp4": QZ_MXFP4, "nvfp4": QZ_NVFP4, "int4": QZ_INT4}
GRANULARITIES = {"tensor": QZ_GRAN_TENSOR, "row": QZ_GRAN_ROW, "block": QZ_GRAN_BLOCK,
                 "unit": QZ_GRAN_UNIT}
BLOCK_SIZE = {QZ_MXFP4: 32, QZ_NVFP4: 16, QZ_INT4: 32}  # INT4: the default group

# Names of the exported C symbols (the whole ABI of include/qz.h).
ABI_SYMBOLS = ("qz_status_string", "qz_workspace_size", "qz_workspace_init", "qz_amax",
               "qz_quantize", "qz_quantize_delayed", "qz_dequantize", "qz_error_stats",
               "qz_error_stats_noalloc", "qz_error_stats_noalloc_status", "qz_stats_merge", "qz_dequantize_asym4", "qz_quant_dot",
               "qz_selftest_pipeline_timeout", "qz_get_device_status", "qz_host_plan_create",
               "qz_host_run", "qz_host_plan_status", "qz_host_plan_destroy")
QZ_HOST_MAX_RUNS = 16


class QzDesc(C.Structure):
    _fields_ = [("format", C.c_int32), ("in_dtype", C.c_int32), ("granularity", C.c_int32),
                ("block_size", C.c_int32), ("elem_round", C.c_int32),
                ("scale_round", C.c_int32), ("rows", C.c_int64), ("cols", C.c_int64),
                ("ld", C.c_int64)]


class QzStats(C.Structure):
    _fields_ = [("sum_sq_err", C.c_double), ("mse", C.c_double),
                ("max_rel_err", C.c_float), ("max_abs_err", C.c_float), ("n", C.c_uint64)]


STATS_BYTES = C.sizeof(QzStats)


class QzHostIo(C.Structure):
    """qz_host_io: one run's device outputs and host copies (0 / None = absent)."""
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p), ("tensor_scale", C.c_void_p),
                ("y", C.c_void_p), ("stats", C.c_void_p), ("codes_host", C.c_void_p),
                ("scales_host", C.c_void_p), ("tensor_scale_host", C.c_void_p),
                ("stats_host", C.c_void_p)]


class QzError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {qz_status_string(status)} (status {status})")
        self.status = status


_lib = None


def lib():
    """The loaded libqz.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        L = C.CDLL(LIB_PATH)
        vp, dp, i32 = C.c_void_p, C.POINTER(QzDesc), C.c_int32
        sig = {
            "qz_status_string": (C.c_char_p, [i32]),
            "qz_workspace_size": (C.c_size_t, [dp]),
            "qz_workspace_init": (i32, [vp, C.c_size_t, vp]),
            "qz_amax": (i32, [dp, vp, vp, vp, vp]),
            "qz_quantize": (i32, [dp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "qz_quantize_delayed": (i32, [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
            "qz_dequantize": (i32, [dp, vp, vp, vp, vp, i32, vp]),
            "qz_error_stats": (i32, [dp, vp, vp, vp, vp, vp, vp, vp]),
            "qz_error_stats_noalloc": (i32, [dp, vp, vp, vp, vp, vp, vp]),
            "qz_error_stats_noalloc_status": (i32, [C.POINTER(C.c_uint32), vp]),
            "qz_stats_merge": (i32, [vp, C.c_int64, vp, vp]),
            "qz_get_device_status": (i32, [vp, C.POINTER(C.c_uint32), vp]),
            "qz_dequantize_asym4": (i32, [vp, vp, vp, C.c_int64, C.c_int64, C.c_int64, vp,
                                          C.c_int64, i32, vp]),
            "qz_selftest_pipeline_timeout": (i32, [vp, C.c_uint64, vp]),
            "qz_quant_dot": (i32, [vp, vp, vp, C.c_int64, C.c_int64, C.c_int64, vp, C.c_int64,
                                   C.c_int64, vp, C.c_int64, vp]),
            "qz_host_plan_create": (i32, [dp, i32, C.c_int64, i32, i32, C.POINTER(vp)]),
            "qz_host_run": (i32, [vp, vp, C.POINTER(QzHostIo)]),
            "qz_host_plan_status": (i32, [vp, C.POINTER(C.c_uint32)]),
            "qz_host_plan_destroy": (None, [vp]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype, f.argtypes = res, args
        _lib = L
    return _lib


# ---------------------------------------------------------------- C ABI, one to one
def qz_status_string(status: int) -> str:
    return lib().qz_status_string(status).decode()


def qz_workspace_size(desc: QzDesc | None = None) -> int:
    return lib().qz_workspace_size(None if desc is None else C.byref(desc))


def qz_workspace_init(ws: int, nbytes: int, stream: int = 0) -> int:
    return lib().qz_workspace_init(ws, nbytes, stream)


def qz_amax(desc: QzDesc, x: int, amax_dev: int, ws: int, stream: int = 0) -> int:
    return lib().qz_amax(C.byref(desc), x, amax_dev, ws, stream)


def qz_quantize(desc: QzDesc, x: int, codes: int, scales: int | None,
                tensor_scale_dev: int | None, tensor_amax_dev: int | None,
                stats_dev: int | None, ws: int | None, stream: int = 0) -> int:
    return lib().qz_quantize(C.byref(desc), x, codes, scales, tensor_scale_dev,
                             tensor_amax_dev, stats_dev, ws, stream)


def qz_quantize_delayed(desc: QzDesc, x: int, codes: int, scales: int | None,
                        tensor_scale_dev: int | None, amax_in_dev: int | None, amax_out_dev: int,
                        stats_dev: int | None, ws: int, stream: int = 0) -> int:
    return lib().qz_quantize_delayed(C.byref(desc), x, codes, scales, tensor_scale_dev,
                                     amax_in_dev, amax_out_dev, stats_dev, ws, stream)


def qz_dequantize_asym4(w: int, scales: int, shifts: int, rows: int, cols: int, group: int,
                        y: int, ld: int, out_dtype: int, stream: int = 0) -> int:
    return lib().qz_dequantize_asym4(w, scales, shifts, rows, cols, group, y, ld, out_dtype,
                                     stream)


def qz_host_plan_create(runs, chunk_rows: int, out_dtype: int, fuse_stats: bool):
    """runs: sequence of QzDesc.  Returns (status, plan handle or None)."""
    arr = (QzDesc * len(runs))(*runs) if len(runs) else None
    h = C.c_void_p()
    st = lib().qz_host_plan_create(arr, len(runs), chunk_rows, out_dtype, int(bool(fuse_stats)),
                                   C.byref(h))
    return st, (h.value if st == QZ_OK else None)


def qz_host_run(plan: int, x_host: int | None, io) -> int:
    """io: sequence of QzHostIo, one per run of the plan."""
    arr = (QzHostIo * len(io))(*io)
    return lib().qz_host_run(plan, x_host, arr)


def qz_host_plan_status(plan: int):
    flags = C.c_uint32(0)
    st = lib().qz_host_plan_status(plan, C.byref(flags))
    return st, flags.value


def qz_host_plan_destroy(plan: int | None) -> None:
    lib().qz_host_plan_destroy(plan)


def qz_quant_dot(w: int, scales: int, shifts: int, n0: int, mid: int, group: int, y: int,
                 ld_y: int, n1: int, z: int, ld_z: int, stream: int = 0) -> int:
    return lib().qz_quant_dot(w, scales, shifts, n0, mid, group, y, ld_y, n1, z, ld_z, stream)


def quant_dot(w, scales, shifts, group: int, y, out=None, stream=None):
    """z = sum_l sc (w - sh) y (see qz_quant_dot): w int32/uint32 CUDA tensor [n0, mid/8],
    scales fp32 [n0, mid/group], shifts int32/uint32 [n0, ceil(mid/group/8)], y bf16
    [mid, n1] (any n1: up to 8 columns stream the weights once, more run on the tcgen05
    tensor cores).  Returns fp32 [n0, n1]."""
    torch = _torch()
    n0, wpr = w.shape
    mid, n1 = y.shape
    if mid != wpr * 8:
        raise ValueError("y must have mid = 8 * w.shape[1] rows")
    z = out if out is not None else torch.empty((n0, n1), dtype=torch.float32, device=w.device)
    _check(qz_quant_dot(w.data_ptr(), scales.data_ptr(), shifts.data_ptr(), n0, mid, group,
                        y.data_ptr(), y.stride(0), n1, z.data_ptr(), z.stride(0),
                        _stream(stream)), "qz_quant_dot")
    return z


def qz_selftest_pipeline_timeout(ws: int, limit_ns: int, stream: int = 0) -> int:
    return lib().qz_selftest_pipeline_timeout(ws, limit_ns, stream)


def qz_dequantize(desc: QzDesc, codes: int, scales: int | None, tensor_scale_dev: int | None,
                  y: int, out_dtype: int, stream: int = 0) -> int:
    return lib().qz_dequantize(C.byref(desc), codes, scales, tensor_scale_dev, y, out_dtype,
                               stream)


def qz_error_stats(desc: QzDesc, x: int, codes: int, scales: int | None,
                   tensor_scale_dev: int | None, stats_dev: int, ws: int,
                   stream: int = 0) -> int:
    return lib().qz_error_stats(C.byref(desc), x, codes, scales, tensor_scale_dev, stats_dev,
                                ws, stream)


def qz_error_stats_noalloc(desc: QzDesc, x: int, codes: int, scales: int | None,
                           tensor_scale_dev: int | None, stats_dev: int, stream: int = 0) -> int:
    """qz_error_stats for callers that cannot allocate: no workspace argument (the library
    uses a fixed scratch array of its own; see include/qz.h)."""
    return lib().qz_error_stats_noalloc(C.byref(desc), x, codes, scales, tensor_scale_dev,
                                        stats_dev, stream)


def qz_error_stats_noalloc_status(stream: int = 0) -> tuple[int, int]:
    """(status, flags): the QZ_FLAG_* bits qz_error_stats_noalloc calls on the current device
    raised since the last query, read and cleared in order on `stream`."""
    flags = C.c_uint32(0)
    st = lib().qz_error_stats_noalloc_status(C.byref(flags), stream)
    return st, flags.value


def qz_stats_merge(parts: int, count: int, out: int, stream: int = 0) -> int:
    return lib().qz_stats_merge(parts, count, out, stream)


def qz_get_device_status(ws: int, stream: int = 0) -> tuple[int, int]:
    flags = C.c_uint32(0)
    st = lib().qz_get_device_status(ws, C.byref(flags), stream)
    return st, flags.value


# ---------------------------------------------------------------- torch marshalling
def _torch():
    import torch
    return torch


def _check(status: int, what: str):
    if status != QZ_OK:
        raise QzError(status, what)


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def _gran(g) -> int:
    return GRANULARITIES[g] if isinstance(g, str) else int(g)


def default_granularity(fmt: int) -> int:
    return QZ_GRAN_BLOCK if fmt in (QZ_MXFP4, QZ_NVFP4, QZ_INT4) else QZ_GRAN_TENSOR


def _dtype_code(dt) -> int:
    torch = _torch()
    if dt == torch.bfloat16:
        return QZ_BF16
    if dt == torch.float32:
        return QZ_F32
    raise TypeError(f"unsupported dtype {dt}: bf16 or fp32")


def make_desc(fmt, in_dtype: int, granularity, rows: int, cols: int, ld: int | None = None,
              scale_round: int = QZ_SCALE_UP, block_size: int | None = None) -> QzDesc:
    """block_size: the INT4 group (16, 32, 64, 128; default 32); fixed by the format else."""
    f = _fmt(fmt)
    bs = block_size if (f == QZ_INT4 and block_size is not None) else BLOCK_SIZE.get(f, 0)
    return QzDesc(f, in_dtype, _gran(granularity), bs, QZ_ROUND_RNE,
                  scale_round, rows, cols, cols if ld is None else ld)


def _rows_cols_ld(t):
    if t.dim() != 2:
        raise ValueError("2-D tensors only")
    rows, cols = t.shape
    if rows and cols and t.stride(1) != 1:
        raise ValueError("the inner dimension must be contiguous")
    ld = t.stride(0) if rows > 1 else cols
    return rows, cols, max(ld, cols)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


class Workspace:
    """Device workspace of qz_workspace_size() bytes, zeroed once (the calls keep it valid)."""

    def __init__(self, device=None):
        torch = _torch()
        self.nbytes = qz_workspace_size()
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device or "cuda")

    @property
    def ptr(self) -> int:
        return self.buf.data_ptr()

    def status(self, stream=None) -> int:
        st, flags = qz_get_device_status(self.ptr, _stream(stream))
        _check(st, "qz_get_device_status")
        return flags

    def clear(self, stream=None):
        _check(qz_workspace_init(self.ptr, self.nbytes, _stream(stream)), "qz_workspace_init")


@dataclass
class Quantized:
    codes: object          # uint8 [rows, cols] or [rows, cols/2]
    scales: object         # fp32 [rows] (ROW), uint8 [rows, cols/bs] (FP4),
                           # fp32 [rows, cols/bs] (INT4), or None
    tensor_scale: object   # fp32 [1]
    fmt: int
    granularity: int
    scale_round: int
    rows: int
    cols: int
    block_size: int = 0    # the INT4 group (0: the format's own block)


@dataclass
class Stats:
    sum_sq_err: float
    mse: float
    max_rel_err: float
    max_abs_err: float
    n: int


def stats_from_bytes(b: bytes) -> Stats:
    return Stats(*struct.unpack("<ddffQ", bytes(b)))


def read_stats(t) -> Stats:
    """Copy a device qz_stats buffer (uint8[STATS_BYTES]) to the host."""
    return stats_from_bytes(t.cpu().numpy().tobytes())


def alloc_outputs(fmt: int, granularity: int, rows: int, cols: int, device,
                  block_size: int | None = None):
    torch = _torch()
    bs = block_size if (fmt == QZ_INT4 and block_size is not None) else BLOCK_SIZE.get(fmt, 0)
    codes = torch.empty((rows, cols // 2 if bs else cols), dtype=torch.uint8, device=device)
    if bs:
        scales = torch.empty((rows, cols // bs),
                             dtype=torch.float32 if fmt == QZ_INT4 else torch.uint8, device=device)
    elif granularity == QZ_GRAN_ROW:
        scales = torch.empty((rows,), dtype=torch.float32, device=device)
    else:
        scales = None
    tscale = torch.empty((1,), dtype=torch.float32, device=device)
    return codes, scales, tscale


def quantize(x, fmt, granularity=None, scale_round: int = QZ_SCALE_UP, tensor_amax=None,
             stats: bool = False, workspace: Workspace | None = None, out=None, stream=None,
             block_size: int | None = None):
    """Quantize a 2-D bf16 / fp32 CUDA tensor.  Returns (Quantized, stats tensor or None).

    tensor_amax: optional fp32 CUDA tensor [1] with alpha (per-tensor / NVFP4 global amax).
    out: optional (codes, scales, tensor_scale) buffers to write into.
    """
    torch = _torch()
    f = _fmt(fmt)
    g = default_granularity(f) if granularity is None else _gran(granularity)
    rows, cols, ld = _rows_cols_ld(x)
    desc = make_desc(f, _dtype_code(x.dtype), g, rows, cols, ld, scale_round, block_size)
    codes, scales, tscale = out if out is not None else alloc_outputs(f, g, rows, cols, x.device,
                                                                      desc.block_size)
    st = torch.empty((STATS_BYTES,), dtype=torch.uint8, device=x.device) if stats else None
    need_ws = stats or (tensor_amax is None and (g == QZ_GRAN_TENSOR or
                                                 (f == QZ_NVFP4 and g == QZ_GRAN_BLOCK)))
    if need_ws and workspace is None:
        workspace = Workspace(x.device)
    rc = qz_quantize(desc, x.data_ptr(), codes.data_ptr(), _ptr(scales), tscale.data_ptr(),
                     _ptr(tensor_amax), _ptr(st), workspace.ptr if workspace else None,
                     _stream(stream))
    _check(rc, "qz_quantize")
    return Quantized(codes, scales, tscale, f, g, scale_round, rows, cols, desc.block_size), st


def quantize_delayed(x, fmt, amax_in, granularity=None, scale_round: int = QZ_SCALE_UP,
                     stats: bool = False, workspace: Workspace | None = None, out=None,
                     amax_out=None, stream=None, block_size: int | None = None):
    """Quantize with the per-tensor scale of an earlier tensor's amax (amax_in: fp32 CUDA
    tensor [1], or None where the granularity needs none) and return this tensor's amax.
    Returns (Quantized, stats tensor or None, amax_out tensor [1])."""
    torch = _torch()
    f = _fmt(fmt)
    g = default_granularity(f) if granularity is None else _gran(granularity)
    rows, cols, ld = _rows_cols_ld(x)
    desc = make_desc(f, _dtype_code(x.dtype), g, rows, cols, ld, scale_round, block_size)
    codes, scales, tscale = out if out is not None else alloc_outputs(f, g, rows, cols, x.device,
                                                                      desc.block_size)
    st = torch.empty((STATS_BYTES,), dtype=torch.uint8, device=x.device) if stats else None
    workspace = workspace or Workspace(x.device)
    amax_out = amax_out if amax_out is not None else torch.empty((1,), dtype=torch.float32,
                                                                 device=x.device)
    rc = qz_quantize_delayed(desc, x.data_ptr(), codes.data_ptr(), _ptr(scales),
                             tscale.data_ptr(), _ptr(amax_in), amax_out.data_ptr(), _ptr(st),
                             workspace.ptr, _stream(stream))
    _check(rc, "qz_quantize_delayed")
    return (Quantized(codes, scales, tscale, f, g, scale_round, rows, cols, desc.block_size), st,
            amax_out)


def dequantize(q: Quantized, out_dtype=None, out=None, stream=None):
    """x^ = decode(codes) * scale as a bf16 (default) or fp32 CUDA tensor."""
    torch = _torch()
    out_dtype = out_dtype or torch.bfloat16
    y = out if out is not None else torch.empty((q.rows, q.cols), dtype=out_dtype,
                                                device=q.codes.device)
    rows, cols, ld = _rows_cols_ld(y)
    desc = make_desc(q.fmt, QZ_BF16, q.granularity, q.rows, q.cols, ld, q.scale_round,
                     q.block_size or None)
    rc = qz_dequantize(desc, q.codes.data_ptr(), _ptr(q.scales), _ptr(q.tensor_scale),
                       y.data_ptr(), _dtype_code(y.dtype), _stream(stream))
    _check(rc, "qz_dequantize")
    return y


def dequantize_asym4(w, scales, shifts, group: int, out_dtype=None, out=None, stream=None):
    """Asymmetric 4-bit group dequantization y = sc * (w - sh) (see qz_dequantize_asym4):
    w int32/uint32 CUDA tensor [rows, cols/8], scales fp32 [rows, cols/group], shifts
    int32/uint32 [rows, ceil(cols/group/8)].  Returns a bf16 (default) or fp32 tensor."""
    torch = _torch()
    rows, wpr = w.shape
    cols = wpr * 8
    out_dtype = out_dtype or torch.bfloat16
    y = out if out is not None else torch.empty((rows, cols), dtype=out_dtype, device=w.device)
    _, _, ld = _rows_cols_ld(y)
    rc = qz_dequantize_asym4(w.data_ptr(), scales.data_ptr(), shifts.data_ptr(), rows, cols,
                             group, y.data_ptr(), ld, _dtype_code(y.dtype), _stream(stream))
    _check(rc, "qz_dequantize_asym4")
    return y


def error_stats(x, q: Quantized, workspace: Workspace | None = None, stream=None):
    """Error statistics of q against x: a device uint8[STATS_BYTES] qz_stats buffer."""
    torch = _torch()
    rows, cols, ld = _rows_cols_ld(x)
    desc = make_desc(q.fmt, _dtype_code(x.dtype), q.granularity, rows, cols, ld, q.scale_round,
                     q.block_size or None)
    st = torch.empty((STATS_BYTES,), dtype=torch.uint8, device=x.device)
    workspace = workspace or Workspace(x.device)
    rc = qz_error_stats(desc, x.data_ptr(), q.codes.data_ptr(), _ptr(q.scales),
                        _ptr(q.tensor_scale), st.data_ptr(), workspace.ptr, _stream(stream))
    _check(rc, "qz_error_stats")
    return st


def amax(x, workspace: Workspace | None = None, stream=None):
    """Largest |x| as an fp32 CUDA tensor [1]."""
    torch = _torch()
    rows, cols, ld = _rows_cols_ld(x)
    desc = make_desc(QZ_INT8, _dtype_code(x.dtype), QZ_GRAN_TENSOR, rows, cols, ld)
    out = torch.empty((1,), dtype=torch.float32, device=x.device)
    workspace = workspace or Workspace(x.device)
    _check(qz_amax(desc, x.data_ptr(), out.data_ptr(), workspace.ptr, _stream(stream)), "qz_amax")
    return out
