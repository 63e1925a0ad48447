"""Quantize a tensor that sits in host memory, with the host<->device copies overlapped with
the kernels: the binding of the C ABI's host round trip (qz_host_plan_create / qz_host_run,
include/qz.h).

``HostRoundTrip`` is the round trip a caller with host data makes: copy x to the device,
quantize it (with the fused error statistics), dequantize it on the device, and copy the
codes, scales, tensor scale and statistics back to pinned host buffers.  The scheduling --
row chunks copied in on one stream, each chunk quantized and dequantized as soon as it has
landed on a second, its codes and scales copied back on a third, the per-tensor amax
folded from the chunk amaxes once every chunk is in, the chunk statistics merged -- is the
library's own (csrc/qz_host.cu); this class allocates the outputs (torch tensors on the
device, pinned host tensors) and passes their pointers in one C call per round trip.

Codes, scales and tensor scales are bit-identical to quantizing the whole tensor in one
call: scale blocks run along a row and never straddle two chunks, a row scale is a row's
own, and the per-tensor amax is the same maximum.  The statistics equal the whole-tensor
ones (maxima exactly, the sum of squares within the library's 1e-5 bound).
"""
from __future__ import annotations

from . import (QZ_BF16, QZ_F32, QZ_GRAN_TENSOR, QZ_NVFP4, QZ_GRAN_BLOCK, QZ_SCALE_UP, STATS_BYTES,
               QzHostIo, _check, _fmt, _gran, _torch, alloc_outputs, default_granularity, make_desc,
               qz_host_plan_create, qz_host_plan_destroy, qz_host_plan_status, qz_host_run,
               stats_from_bytes)


def needs_tensor_amax(fmt: int, gran: int) -> bool:
    """The format's scale depends on the amax of the whole tensor."""
    return gran == QZ_GRAN_TENSOR or (fmt == QZ_NVFP4 and gran == QZ_GRAN_BLOCK)


def _ptr(t):
    return None if t is None else t.data_ptr()


class HostRoundTrip:
    """A reusable plan for the host round trip of a [rows, cols] tensor.

    runs        list of formats, or of (format, granularity) pairs (granularity None: the
                format's default); each gets codes, scales, tensor scale, statistics and a
                dequantized copy on the device.
    in_dtype    "bf16" or "f32": the dtype of the host tensor handed to ``run``.
    chunk_rows  rows per host-to-device copy.
    out_dtype   dtype of the dequantized tensors ("bf16" or "f32"); they stay on the device
                (``self.y``).
    stats       fuse the error statistics into the quantize calls.

    Device buffers, pinned host outputs and the library's plan (its device copy of x,
    workspace, streams and events) are allocated here, once; ``run`` allocates nothing.
    The host outputs are overwritten by every ``run``.
    """

    def __init__(self, rows: int, cols: int, runs, in_dtype: str = "bf16", chunk_rows: int = 4096,
                 device=None, out_dtype: str = "bf16", stats: bool = True,
                 scale_round: int = QZ_SCALE_UP):
        torch = _torch()
        if chunk_rows <= 0:
            raise ValueError("chunk_rows must be positive")
        self.plan = None
        self.dev = torch.device(device if device is not None else "cuda")
        self.rows, self.cols, self.stats = rows, cols, stats
        self.in_code = QZ_BF16 if in_dtype == "bf16" else QZ_F32
        self.in_torch = torch.bfloat16 if in_dtype == "bf16" else torch.float32
        self.out_code = QZ_BF16 if out_dtype == "bf16" else QZ_F32
        ydt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
        self.runs = []
        for r in runs:
            f, g = (r, None) if not isinstance(r, (tuple, list)) else r
            f = _fmt(f)
            self.runs.append((f, default_granularity(f) if g is None else _gran(g)))
        pin = dict(pin_memory=True)
        self.out, self.y, self.st, self.host, self.io = [], [], [], [], []
        for f, g in self.runs:
            codes, scales, ts = alloc_outputs(f, g, rows, cols, self.dev)
            self.out.append((codes, scales, ts))
            self.y.append(torch.empty((rows, cols), dtype=ydt, device=self.dev))
            self.st.append(torch.empty((STATS_BYTES,), dtype=torch.uint8, device=self.dev))
            h = dict(
                codes=torch.empty(codes.shape, dtype=codes.dtype, **pin),
                scales=None if scales is None else torch.empty(scales.shape, dtype=scales.dtype,
                                                               **pin),
                tensor_scale=torch.empty((1,), dtype=torch.float32, **pin),
                stats=torch.empty((STATS_BYTES,), dtype=torch.uint8, **pin))
            self.host.append(h)
            self.io.append(QzHostIo(
                codes=_ptr(codes), scales=_ptr(scales), tensor_scale=_ptr(ts),
                y=_ptr(self.y[-1]), stats=_ptr(self.st[-1]) if stats else None,
                codes_host=_ptr(h["codes"]), scales_host=_ptr(h["scales"]),
                tensor_scale_host=_ptr(h["tensor_scale"]),
                stats_host=_ptr(h["stats"]) if stats else None))
        descs = [make_desc(f, self.in_code, g, rows, cols, cols, scale_round) for f, g in self.runs]
        with torch.cuda.device(self.dev):
            st, self.plan = qz_host_plan_create(descs, chunk_rows, self.out_code, stats)
        _check(st, "qz_host_plan_create")
        torch.cuda.synchronize(self.dev)

    def run(self, x_host):
        """One round trip of the host tensor x_host ([rows, cols], the plan's dtype,
        contiguous; pinned for overlapped copies).  Returns, per run, the dict of pinned host
        outputs (codes, scales, tensor_scale, stats as a uint8 qz_stats record); the device
        keeps the dequantized tensors in ``self.y``.  Returns when everything is done."""
        if tuple(x_host.shape) != (self.rows, self.cols) or x_host.dtype != self.in_torch:
            raise ValueError("x_host does not match the plan's shape / dtype")
        if not x_host.is_contiguous():
            raise ValueError("x_host must be contiguous")
        if x_host.is_cuda:
            raise ValueError("x_host must be in host memory")
        xp = x_host.data_ptr() if x_host.numel() else None
        _check(qz_host_run(self.plan, xp, self.io), "qz_host_run")
        return self.host

    def status(self) -> int:
        """QZ_FLAG_* bits the plan's calls have raised (sticky)."""
        st, flags = qz_host_plan_status(self.plan)
        _check(st, "qz_host_plan_status")
        return flags

    def read_stats(self, j: int):
        """Statistics of run j from the last ``run`` (host record -> Stats)."""
        return stats_from_bytes(self.host[j]["stats"].numpy().tobytes())

    def bytes_in(self) -> int:
        return self.rows * self.cols * (2 if self.in_code == QZ_BF16 else 4)

    def bytes_out(self) -> int:
        return sum(t.numel() * t.element_size() for h in self.host for t in h.values()
                   if t is not None and (self.stats or t is not h["stats"]))

    def close(self):
        """Free the library's plan (also done when the object is collected)."""
        if self.plan is not None:
            qz_host_plan_destroy(self.plan)
            self.plan = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
