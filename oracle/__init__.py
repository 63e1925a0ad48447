"""Python view of the CPU oracle (ctypes over ``liboracle.so``).

TEST INFRASTRUCTURE ONLY.  The oracle is the plain CPU definition of what the CUDA
library must compute bit for bit: quantize to INT8 / FP8 E4M3 / FP8 E5M2 / MXFP4 / NVFP4 /
INT4, dequantize (also the asymmetric 4-bit group form of the blog's "Puzzles 12"), and the
error statistics, as described in the blog post
"浅谈低精度浮点数" (A brief talk on low-precision floats).  Only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import it.

Tensors are numpy arrays: bf16 data is carried as ``np.uint16`` bit patterns, fp32 as
``np.float32``.  A 2-D input may be a row-strided view (leading dimension > cols).
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np

from . import build as _build

INT8, E4M3, E5M2, MXFP4, NVFP4, INT4 = 1, 2, 3, 4, 5, 6
E2M1, E8M0 = 16, 17
BF16, F32 = 1, 2
GRAN_TENSOR, GRAN_ROW, GRAN_BLOCK, GRAN_UNIT = 1, 2, 3, 4
SCALE_UP, SCALE_NEAREST = 0, 1
OK, ERR_ARG, ERR_NONFINITE = 0, 1, 2


class OracleError(RuntimeError):
    pass


class _Stats(C.Structure):
    _fields_ = [("sum_sq_err", C.c_double), ("mse", C.c_double),
                ("max_rel_err", C.c_float), ("max_abs_err", C.c_float),
                ("n", C.c_uint64)]


@dataclass
class Stats:
    sum_sq_err: float
    mse: float
    max_rel_err: float
    max_abs_err: float
    n: int


_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        u32, i32, i64, vp, dbl = C.c_uint32, C.c_int, C.c_int64, C.c_void_p, C.c_double
        fp = C.POINTER(C.c_float)
        sp = C.POINTER(_Stats)
        sig = {
            "orc_decode_fp32": (dbl, [u32]),
            "orc_decode_bf16": (dbl, [C.c_uint16]),
            "orc_encode_fp32": (u32, [dbl]),
            "orc_bf16_rne": (C.c_uint16, [u32]),
            "orc_decode_code": (dbl, [i32, u32]),
            "orc_encode_elem": (u32, [i32, u32]),
            "orc_mx_scale_exponent": (i32, [u32, i32]),
            "orc_nv_block_scale_code": (u32, [u32, i32]),
            "orc_amax": (i32, [i32, i64, i64, i64, vp, fp, i32]),
            "orc_quantize": (i32, [i32, i32, i32, i32, i32, i64, i64, i64, vp, vp, vp, fp, fp,
                                   sp, i32]),
            "orc_dequantize": (i32, [i32, i32, i32, i64, i64, i64, vp, vp, fp, vp, i32, i32]),
            "orc_error_stats": (i32, [i32, i32, i32, i32, i64, i64, i64, vp, vp, vp, fp, sp,
                                      i32]),
            "orc_dequant_asym4": (i32, [i64, i64, i64, vp, vp, vp, vp, i32, i32]),
            "orc_quant_dot": (i32, [i64, i64, i64, i64, vp, vp, vp, vp, vp, vp, i32]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


# ---------------------------------------------------------------- scalar helpers
def f32_bits(v) -> int:
    return int(np.array(v, dtype=np.float32).view(np.uint32))


def bits_f32(b: int) -> np.float32:
    return np.array(b, dtype=np.uint32).view(np.float32)[()]


def decode_fp32(bits: int) -> float:
    return lib().orc_decode_fp32(bits)


def decode_bf16(bits: int) -> float:
    return lib().orc_decode_bf16(bits)


def encode_fp32(v: float) -> int:
    return lib().orc_encode_fp32(v)


def bf16_rne(fp32_bits: int) -> int:
    return lib().orc_bf16_rne(fp32_bits)


def decode_code(fmt: int, code: int) -> float:
    return lib().orc_decode_code(fmt, code)


def encode_elem(fmt: int, v) -> int:
    """Element code of the binary32 value v (RNE, saturating, sign-preserving zero)."""
    return lib().orc_encode_elem(fmt, f32_bits(v))


def mx_scale_exponent(t, scale_round: int = SCALE_UP) -> int:
    return lib().orc_mx_scale_exponent(f32_bits(t), scale_round)


def nv_block_scale_code(t, scale_round: int = SCALE_UP) -> int:
    return lib().orc_nv_block_scale_code(f32_bits(t), scale_round)


# ---------------------------------------------------------------- tensor helpers
def _dtype_of(x: np.ndarray) -> int:
    if x.dtype == np.uint16:
        return BF16
    if x.dtype == np.float32:
        return F32
    raise TypeError("x must be np.uint16 (bf16 bits) or np.float32")


def _rows_cols_ld(x: np.ndarray):
    if x.ndim != 2:
        raise ValueError("2-D tensors only")
    rows, cols = x.shape
    isz = x.dtype.itemsize
    if rows and cols and x.strides[1] != isz:
        raise ValueError("inner dimension must be contiguous")
    ld = x.strides[0] // isz if rows > 1 else cols
    return rows, cols, max(ld, cols)


def _ptr(a):
    return None if a is None else a.ctypes.data


def _check(rc: int, what: str):
    if rc != OK:
        raise OracleError(f"{what}: oracle returned {rc}")


def code_bytes(fmt: int, rows: int, cols: int) -> int:
    return rows * cols // 2 if fmt in (MXFP4, NVFP4, INT4) else rows * cols


def block_of(fmt: int, block_size: int | None = None) -> int:
    """Block (group) size: fixed for MXFP4 / NVFP4, chosen for INT4 (default 32)."""
    if fmt == INT4:
        return 32 if block_size is None else block_size
    return {MXFP4: 32, NVFP4: 16}.get(fmt, 0)


def amax(x: np.ndarray, nthreads: int = 0) -> float:
    rows, cols, ld = _rows_cols_ld(x)
    out = C.c_float(0)
    _check(lib().orc_amax(_dtype_of(x), rows, cols, ld, _ptr(x), C.byref(out), nthreads),
           "amax")
    return np.float32(out.value)


def quantize(x: np.ndarray, fmt: int, granularity: int, scale_round: int = SCALE_UP,
             tensor_amax=None, stats: bool = False, nthreads: int = 0,
             block_size: int | None = None):
    """Return (codes uint8, scales, tensor_scale float32, Stats or None).

    codes: [rows, cols] (8-bit formats) or [rows, cols/2] (4-bit, low nibble first);
    scales: float32 [rows] for ROW, uint8 [rows, cols/bs] for MXFP4/NVFP4, float32
    [rows, cols/bs] for INT4, else None.
    """
    rows, cols, ld = _rows_cols_ld(x)
    bs = block_of(fmt, block_size)
    codes = np.zeros((rows, cols // 2 if bs else cols), dtype=np.uint8)
    if bs:
        scales = np.zeros((rows, cols // bs if bs else 0),
                          dtype=np.float32 if fmt == INT4 else np.uint8)
    elif granularity == GRAN_ROW:
        scales = np.zeros((rows,), dtype=np.float32)
    else:
        scales = None
    ts = C.c_float(0)
    ta = None if tensor_amax is None else C.c_float(float(tensor_amax))
    st = _Stats() if stats else None
    rc = lib().orc_quantize(fmt, _dtype_of(x), granularity, bs, scale_round, rows, cols, ld,
                            _ptr(x), _ptr(codes), _ptr(scales), C.byref(ts),
                            None if ta is None else C.byref(ta),
                            None if st is None else C.byref(st), nthreads)
    _check(rc, "quantize")
    s = None if st is None else Stats(st.sum_sq_err, st.mse, np.float32(st.max_rel_err),
                                      np.float32(st.max_abs_err), int(st.n))
    return codes, scales, np.float32(ts.value), s


def dequantize(codes: np.ndarray, scales, tensor_scale, fmt: int, granularity: int,
               rows: int, cols: int, out_dtype: int = BF16, nthreads: int = 0,
               block_size: int | None = None):
    bs = block_of(fmt, block_size)
    y = np.zeros((rows, cols), dtype=np.uint16 if out_dtype == BF16 else np.float32)
    ts = C.c_float(float(tensor_scale if tensor_scale is not None else 1.0))
    rc = lib().orc_dequantize(fmt, granularity, bs, rows, cols, cols, _ptr(codes),
                              _ptr(scales), C.byref(ts), _ptr(y), out_dtype, nthreads)
    _check(rc, "dequantize")
    return y


def error_stats(x: np.ndarray, codes: np.ndarray, scales, tensor_scale, fmt: int,
                granularity: int, nthreads: int = 0, block_size: int | None = None) -> Stats:
    rows, cols, ld = _rows_cols_ld(x)
    bs = block_of(fmt, block_size)
    ts = C.c_float(float(tensor_scale if tensor_scale is not None else 1.0))
    st = _Stats()
    rc = lib().orc_error_stats(fmt, _dtype_of(x), granularity, bs, rows, cols, ld, _ptr(x),
                               _ptr(codes), _ptr(scales), C.byref(ts), C.byref(st),
                               nthreads)
    _check(rc, "error_stats")
    return Stats(st.sum_sq_err, st.mse, np.float32(st.max_rel_err),
                 np.float32(st.max_abs_err), int(st.n))


def dequant_asym4(w: np.ndarray, scales: np.ndarray, shifts: np.ndarray, rows: int, cols: int,
                  group: int, out_dtype: int = F32, nthreads: int = 0):
    """Asymmetric 4-bit group dequantization of the "Puzzles 12" section:
    y = sc * (w - sh).  w: uint32 [rows, cols/8]; scales: float32 [rows, cols/group];
    shifts: uint32 [rows, ceil(cols/group/8)]; nibbles low first.  Returns y as bf16 bits
    (uint16) or float32."""
    y = np.zeros((rows, cols), dtype=np.uint16 if out_dtype == BF16 else np.float32)
    w = np.ascontiguousarray(w, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    shifts = np.ascontiguousarray(shifts, dtype=np.uint32)
    rc = lib().orc_dequant_asym4(rows, cols, group, _ptr(w), _ptr(scales), _ptr(shifts),
                                 _ptr(y), out_dtype, nthreads)
    _check(rc, "dequant_asym4")
    return y


def quant_dot(w: np.ndarray, scales: np.ndarray, shifts: np.ndarray, y_bf16: np.ndarray,
              group: int, nthreads: int = 0):
    """The puzzle's z = sum_l sc (w - sh) y, in double: returns (z, sum of |terms|), both
    float64 [n0, n1].  w uint32 [n0, mid/8]; scales float32 [n0, mid/group]; shifts uint32
    [n0, ceil(mid/group/8)]; y bf16 bits uint16 [mid, n1]."""
    n0, wpr = w.shape
    mid = wpr * 8
    n1 = y_bf16.shape[1]
    z = np.zeros((n0, n1), dtype=np.float64)
    za = np.zeros((n0, n1), dtype=np.float64)
    w = np.ascontiguousarray(w, dtype=np.uint32)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    shifts = np.ascontiguousarray(shifts, dtype=np.uint32)
    y_bf16 = np.ascontiguousarray(y_bf16, dtype=np.uint16)
    rc = lib().orc_quant_dot(n0, mid, group, n1, _ptr(w), _ptr(scales), _ptr(shifts),
                             _ptr(y_bf16), _ptr(z), _ptr(za), nthreads)
    _check(rc, "quant_dot")
    return z, za
