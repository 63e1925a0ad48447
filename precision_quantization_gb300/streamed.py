"""Quantize a tensor that sits in pinned host memory, with the host<->device copies
overlapped with the kernels.

``HostRoundTrip`` is the round trip a caller with host data makes: copy x to the device,
quantize it (with the fused error statistics), dequantize it on the device, and copy the
codes, scales, tensor scale and statistics back to pinned host buffers.  The rows go over
in chunks on a copy stream, so the kernels of chunk i run while chunk i + 1 is in flight
and the results of chunk i travel back while later chunks arrive.  Every step of the
computation is one of the C ABI calls of ``include/qz.h``; this module only schedules them
on three CUDA streams:

* in-stream: host-to-device copies of the row chunks of x;
* kernel stream: for each chunk, as soon as it has landed, the formats whose scales are
  local to a row or a block (MXFP4 / NVFP4 UNIT, ROW, UNIT) are quantized and dequantized,
  and, when some format needs a per-tensor scale, the chunk's amax is taken (qz_amax).
  Once every chunk is in, the chunk amaxes are folded by one more qz_amax over them (the
  largest of non-negative values is their amax), and the formats with a per-tensor scale
  (TENSOR, NVFP4 BLOCK) are quantized chunk by chunk with that amax supplied.  The
  statistics of the chunks are folded with qz_stats_merge;
* out-stream: device-to-host copies of each chunk's codes and scales once its kernels are
  done, then the tensor scale and the statistics.

Codes, scales and tensor scales are bit-identical to quantizing the whole tensor in one
call: scale blocks run along a row and never straddle two chunks, a row scale is a row's
own, and the per-tensor amax is the same maximum.  The statistics equal the whole-tensor
ones (maxima exactly, the sum of squares within the library's 1e-5 bound).
"""
from __future__ import annotations

from . import (QZ_BF16, QZ_F32, QZ_GRAN_BLOCK, QZ_GRAN_TENSOR, QZ_INT8, QZ_NVFP4, QZ_SCALE_UP,
               STATS_BYTES, Workspace, _check, _fmt, _gran, _torch, alloc_outputs,
               default_granularity, make_desc, qz_amax, qz_dequantize, qz_quantize,
               qz_stats_merge, stats_from_bytes)


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

    Device buffers, pinned host outputs, streams and events are allocated here, once;
    ``run`` allocates nothing.  The host outputs are overwritten by every ``run``.
    """

    def __init__(self, rows: int, cols: int, runs, in_dtype: str = "bf16", chunk_rows: int = 4096,
                 device=None, out_dtype: str = "bf16", stats: bool = True,
                 scale_round: int = QZ_SCALE_UP):
        torch = _torch()
        if chunk_rows <= 0:
            raise ValueError("chunk_rows must be positive")
        self.dev = torch.device(device if device is not None else "cuda")
        self.rows, self.cols, self.stats = rows, cols, stats
        self.in_code = QZ_BF16 if in_dtype == "bf16" else QZ_F32
        tdt = torch.bfloat16 if in_dtype == "bf16" else torch.float32
        self.out_code = QZ_BF16 if out_dtype == "bf16" else QZ_F32
        ydt = torch.bfloat16 if out_dtype == "bf16" else torch.float32
        self.chunks = [(r0, min(rows, r0 + chunk_rows)) for r0 in range(0, rows, chunk_rows)]
        k = len(self.chunks)
        self.runs = []
        for r in runs:
            f, g = (r, None) if not isinstance(r, (tuple, list)) else r
            f = _fmt(f)
            self.runs.append((f, default_granularity(f) if g is None else _gran(g)))
        self.x = torch.empty((rows, cols), dtype=tdt, device=self.dev)
        self.ws = Workspace(self.dev)
        pin = dict(pin_memory=True)
        self.out, self.y, self.parts, self.st, self.host = [], [], [], [], []
        self.desc = []  # per run: one descriptor per chunk
        for f, g in self.runs:
            codes, scales, ts = alloc_outputs(f, g, rows, cols, self.dev)
            self.out.append((codes, scales, ts))
            self.y.append(torch.empty((rows, cols), dtype=ydt, device=self.dev))
            self.parts.append(torch.empty((max(k, 1), STATS_BYTES), dtype=torch.uint8,
                                          device=self.dev))
            self.st.append(torch.empty((STATS_BYTES,), dtype=torch.uint8, device=self.dev))
            self.host.append(dict(
                codes=torch.empty(codes.shape, dtype=codes.dtype, **pin),
                scales=None if scales is None else torch.empty(scales.shape, dtype=scales.dtype,
                                                               **pin),
                tensor_scale=torch.empty((1,), dtype=torch.float32, **pin),
                stats=torch.empty((STATS_BYTES,), dtype=torch.uint8, **pin)))
            self.desc.append([make_desc(f, self.in_code, g, r1 - r0, cols, cols, scale_round)
                              for r0, r1 in self.chunks])
        self.whole = [make_desc(f, self.in_code, g, rows, cols, cols, scale_round)
                      for f, g in self.runs]
        self.need_alpha = any(needs_tensor_amax(f, g) for f, g in self.runs)
        self.amax_desc = [make_desc(QZ_INT8, self.in_code, QZ_GRAN_TENSOR, r1 - r0, cols)
                          for r0, r1 in self.chunks]
        self.fold_desc = make_desc(QZ_INT8, QZ_F32, QZ_GRAN_TENSOR, 1, max(k, 1))
        self.amax_parts = torch.zeros((max(k, 1),), dtype=torch.float32, device=self.dev)
        self.alpha = torch.empty((1,), dtype=torch.float32, device=self.dev)
        self.s_in = torch.cuda.Stream(self.dev)
        self.s_k = torch.cuda.Stream(self.dev)
        self.s_out = torch.cuda.Stream(self.dev)
        self.ev_in = [torch.cuda.Event() for _ in self.chunks]
        self.ev_run = [[torch.cuda.Event() for _ in self.chunks] for _ in self.runs]
        self.ev_end = torch.cuda.Event()
        torch.cuda.synchronize(self.dev)

    def _quant_chunk(self, j: int, i: int, amax_ptr):
        """Quantize (+ statistics) and dequantize chunk i of run j on the kernel stream."""
        r0, r1 = self.chunks[i]
        codes, scales, ts = self.out[j]
        d = self.desc[j][i]
        sk = self.s_k.cuda_stream
        cs = codes[r0:r1]
        ss = None if scales is None else scales[r0:r1]
        st = self.parts[j][i].data_ptr() if self.stats else None
        _check(qz_quantize(d, self.x[r0:r1].data_ptr(), cs.data_ptr(), _ptr(ss), ts.data_ptr(),
                           amax_ptr, st, self.ws.ptr, sk), "qz_quantize")
        _check(qz_dequantize(d, cs.data_ptr(), _ptr(ss), ts.data_ptr(),
                             self.y[j][r0:r1].data_ptr(), self.out_code, sk), "qz_dequantize")
        self.ev_run[j][i].record(self.s_k)
        # the chunk's codes and scales go back as soon as they exist
        torch = _torch()
        self.s_out.wait_event(self.ev_run[j][i])
        with torch.cuda.stream(self.s_out):
            h = self.host[j]
            h["codes"][r0:r1].copy_(cs, non_blocking=True)
            if ss is not None:
                h["scales"][r0:r1].copy_(ss, non_blocking=True)

    def run(self, x_host):
        """One round trip of the pinned host tensor x_host ([rows, cols], the plan's dtype,
        contiguous).  Returns, per run, the dict of pinned host outputs (codes, scales,
        tensor_scale, stats as a uint8 qz_stats record); the device keeps the dequantized
        tensors in ``self.y``.  Synchronises the plan's streams before it returns."""
        torch = _torch()
        if tuple(x_host.shape) != (self.rows, self.cols) or x_host.dtype != self.x.dtype:
            raise ValueError("x_host does not match the plan's shape / dtype")
        if not x_host.is_contiguous():
            raise ValueError("x_host must be contiguous")
        sk = self.s_k.cuda_stream
        if not self.chunks:  # empty tensor: one call per run writes its scale and statistics
            for j in range(len(self.runs)):
                codes, scales, ts = self.out[j]
                _check(qz_quantize(self.whole[j], self.x.data_ptr(), codes.data_ptr(),
                                   _ptr(scales), ts.data_ptr(), None,
                                   self.st[j].data_ptr() if self.stats else None, self.ws.ptr,
                                   sk), "qz_quantize")
        with torch.cuda.stream(self.s_in):
            for i, (r0, r1) in enumerate(self.chunks):
                self.x[r0:r1].copy_(x_host[r0:r1], non_blocking=True)
                self.ev_in[i].record(self.s_in)
        local = [j for j, (f, g) in enumerate(self.runs) if not needs_tensor_amax(f, g)]
        tensor = [j for j, (f, g) in enumerate(self.runs) if needs_tensor_amax(f, g)]
        for i, (r0, r1) in enumerate(self.chunks):
            self.s_k.wait_event(self.ev_in[i])
            for j in local:
                self._quant_chunk(j, i, None)
            if self.need_alpha:
                _check(qz_amax(self.amax_desc[i], self.x[r0:r1].data_ptr(),
                               self.amax_parts[i:i + 1].data_ptr(), self.ws.ptr, sk), "qz_amax")
        if self.need_alpha and self.chunks:
            _check(qz_amax(self.fold_desc, self.amax_parts.data_ptr(), self.alpha.data_ptr(),
                           self.ws.ptr, sk), "qz_amax")
            for i in range(len(self.chunks)):
                for j in tensor:
                    self._quant_chunk(j, i, self.alpha.data_ptr())
        if self.stats and self.chunks:
            for j in range(len(self.runs)):
                _check(qz_stats_merge(self.parts[j].data_ptr(), len(self.chunks),
                                      self.st[j].data_ptr(), sk), "qz_stats_merge")
        self.ev_end.record(self.s_k)
        self.s_out.wait_event(self.ev_end)
        with torch.cuda.stream(self.s_out):
            for j in range(len(self.runs)):
                self.host[j]["tensor_scale"].copy_(self.out[j][2], non_blocking=True)
                if self.stats:
                    self.host[j]["stats"].copy_(self.st[j], non_blocking=True)
        self.s_out.synchronize()
        self.s_k.synchronize()
        return self.host

    def read_stats(self, j: int):
        """Statistics of run j from the last ``run`` (host record -> Stats)."""
        return stats_from_bytes(self.host[j]["stats"].numpy().tobytes())

    def bytes_in(self) -> int:
        return self.x.numel() * self.x.element_size()

    def bytes_out(self) -> int:
        return sum(t.numel() * t.element_size() for h in self.host for t in h.values()
                   if t is not None and (self.stats or t is not h["stats"]))
