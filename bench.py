"""Throughput of the quantize -> dequantize round trip (with the fused error statistics) on
the large streaming workload: 32768 x 8192 bf16, |x| = exp(N(0, 2^2)) with random sign,
to MXFP4 and to NVFP4.

One step = MXFP4 quantize (+ error stats) -> dequantize (bf16), then NVFP4 amax ->
quantize (+ error stats) -> dequantize (bf16): 5 kernel launches over inputs already in
HBM.  The metric is GB/s of algorithmic bytes (bytes in + bytes out of every kernel of
the step) per second of device time, and elements/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own replica on its own
GPU (the path has no exchange step), timing is max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "quantize/dequant GB/s (bytes in+out), % of GB300 HBM peak, per format"
ROWS, COLS = 32768, 8192
WORKLOAD = "lognormal-stream-32768x8192-bf16"
L2_FLUSH_BYTES = 256 << 20
KERNEL_SOURCES = ["precision_quantization_gb300/csrc/qz_device.cuh",
                  "precision_quantization_gb300/csrc/qz_pipe.cuh",
                  "precision_quantization_gb300/csrc/qz_quant4.cu",
                  "precision_quantization_gb300/csrc/qz_dequant.cu",
                  "precision_quantization_gb300/csrc/qz_amax.cu"]


class L2Flush:
    """Empties the L2 of the timed workload's data between timed iterations: a write of
    L2_FLUSH_BYTES (more than the 126 MB L2), then a read of as many other bytes, which
    writes the first buffer's dirty lines back to DRAM before the timed region starts.
    Without the read, the next timed kernel would pay for up to 126 MB of the flush's
    write-back (about 19 us at the copy peak), a cost of the flush, not of the kernel."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty((L2_FLUSH_BYTES,), dtype=torch.uint8, device=dev)
        self.r = torch.zeros((L2_FLUSH_BYTES // 8,), dtype=torch.int64, device=dev)

    def run(self):
        self.w.zero_()
        self.r.max()  # reads every byte of the second buffer


def algorithmic_bytes(n: int) -> dict:
    """Bytes in + bytes out per launch, from the formats' layouts (bf16 input and output,
    E2M1 codes 0.5 B/element, one E8M0 byte per 32 / one E4M3 byte per 16 elements, one
    fp32 tensor scale, one 32-byte stats record)."""
    x = 2 * n
    mx_out = n // 2 + n // 32
    nv_out = n // 2 + n // 16
    return {
        "mx_quant": x + mx_out + 32,
        "mx_dequant": mx_out + x,
        "nv_amax": x + 4,
        "nv_quant": x + 4 + nv_out + 4 + 32,
        "nv_dequant": nv_out + 4 + x,
    }


def source_sha() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured",
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", 1700.0))}
    return {"hbm_gbs": 6800.0, "source": "fallback", "bf16_tflops_sustained": 1700.0}


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    k = d.get("kernels", {}).get(kernel)
    if not k or k.get("source_sha") != source_sha():
        return None
    return k.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) while the timed region runs."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append((time.perf_counter(), ln.strip()))

    def wait_first(self, timeout: float = 10.0):
        t = time.perf_counter()
        while self.proc and not self.lines and time.perf_counter() - t < timeout:
            time.sleep(0.02)

    def window(self, t0: float, t1: float):
        self.t0, self.t1 = t0, t1

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self) -> dict:
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        t0, t1 = getattr(self, "t0", None), getattr(self, "t1", None)
        sel = [ln for (ts, ln) in self.lines if t0 is None or t0 <= ts <= t1 + 0.25]
        if not sel and self.lines:  # region shorter than the sampling period: nearest sample
            sel = [min(self.lines, key=lambda p: abs(p[0] - (t0 or 0)))[1]]
        for ln in sel:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for name, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# Every format of the five named workloads, all at full size, timed per call: quantize with
# the fused error stats (including the in-library amax pass where the scale is per tensor),
# the quantize alone, and dequantize; after an L2 flush (cold), and for the workloads that
# fit the 126 MB L2 in part or whole (1 to 3) also back to back without it (warm).
# "delayed": qz_quantize_delayed, the per-tensor scale from an amax handed in (here the
# tensor's own, computed beforehand) and this tensor's amax returned, in one pass.
MATRIX = [
    (1, None, [("int8", "tensor"), ("e4m3", "tensor"), ("mxfp4", "block"), ("nvfp4", "block")]),
    (2, None, [("int8", "row"), ("e4m3", "row"), ("mxfp4", "block"), ("nvfp4", "block"),
               ("int4", "block", 128), ("asym4", "group", 128), ("qdot", "group", 128, 1),
               ("qdot", "group", 128, 8), ("qdot", "group", 128, 4096)]),
    (3, None, [("e4m3", "row"), ("e5m2", "row"), ("nvfp4", "block"), ("nvfp4", "block", "delayed")]),
    (4, None, [("mxfp4", "block"), ("nvfp4", "block"), ("nvfp4", "block", "delayed"),
               ("int4", "block", 32), ("qdot", "group", 128, 8), ("qdot", "group", 128, 2048)]),
    (5, None, [(f, g) for f in ("int8", "e4m3", "e5m2") for g in ("unit", "tensor")] +
              [(f, g) for f in ("mxfp4", "nvfp4") for g in ("unit", "block")] +
              [("e4m3", "tensor", "delayed"), ("nvfp4", "block", "delayed")]),
]


WARM_WORKLOADS = (1, 2, 3)


def compact_matrix(rows: list) -> dict:
    """One short string per matrix row, "q/qn/dq" fractions of the measured HBM peak
    (quantize with statistics, quantize alone, dequantize; cold L2), then "|q/dq" warm for
    the L2-sized workloads; kept at the end of the JSON line."""
    def f(v):
        return "-" if v is None else f"{v:.3f}".lstrip("0")
    out = {}
    for r in rows:
        key = f"{r.get('workload_id', '?')}:{r['format']}/{r['granularity'].replace(' ', '')}"
        v = f"{f(r.get('quantize_frac'))}/{f(r.get('quantize_nostats_frac'))}/{f(r.get('dequantize_frac'))}"
        if "quantize_warm_frac" in r:
            v += f"|{f(r['quantize_warm_frac'])}/{f(r['dequantize_warm_frac'])}"
        if "tflops" in r:
            v += f" {r['tflops']}TF/s={f(r['tflops_frac'])}"
        out[key] = v
    return out


def make_timed(dev, flush, reps):
    """Mean CUDA-event time (ms) of fn on the current stream over `reps` launches after 3,
    each after an L2 flush unless cold=False."""
    import torch
    stream = torch.cuda.current_stream(dev)

    def timed(fn, cold=True):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            if cold:
                flush.run()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b))
        # the mean: the event clock ticks in steps of about 2 us here, too coarse for the
        # 5-50 us launches of the smaller workloads, and the mean over many launches with
        # varying start phases is not biased by the step the way a median is
        return statistics.mean(ts)
    return timed


# Quantized products on the tensor cores beyond the matrix rows: square and prefill-sized
# shapes, the group sizes with their own decode forms, and a short activation block.
QDOT_SWEEP = [(4096, 4096, 128, 4096), (8192, 8192, 128, 4096), (32768, 8192, 128, 2048),
              (4096, 4096, 64, 4096), (4096, 4096, 32, 4096), (4096, 4096, 128, 512)]


def measure_qdot_sweep(dev, peaks, flush, reps=30) -> list:
    timed = make_timed(dev, flush, reps)
    out = []
    for n0, mid, group, n1 in QDOT_SWEEP:
        row = measure_qdot(f"weight-{n0}x{mid}", n0, mid, group, n1, timed, peaks, dev)
        out.append({k: row[k] for k in ("workload", "granularity", "dequantize_us", "tflops",
                                        "tflops_peak", "tflops_frac")})
    return out


def measure_matrix(dev, peaks, flush, x4=None, reps=30, which=(1, 2, 3, 4, 5), max_rows=None) -> list:
    import numpy as np
    import torch
    import precision_quantization_gb300 as qz
    import workloads as W
    out = []
    stream = torch.cuda.current_stream(dev)
    sp = stream.cuda_stream
    ws = qz.Workspace(dev)
    st = torch.empty((qz.STATS_BYTES,), dtype=torch.uint8, device=dev)
    timed = make_timed(dev, flush, reps)

    for k, rows, runs in MATRIX:
        if k not in which:
            continue
        if max_rows is not None:
            rows = min(max_rows, W.WORKLOADS[k]["rows"])
        if k == 4 and x4 is not None and max_rows is None:
            x_np, x = None, x4
        else:
            x_np = W.workload(k, rows=rows)
            if x_np.dtype == np.uint16:
                x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(dev)
            else:
                x = torch.from_numpy(x_np).to(dev)
        r, c = x.shape
        n = r * c
        eb = x.element_size()
        idt = qz.QZ_BF16 if x.dtype == torch.bfloat16 else qz.QZ_F32
        name = W.WORKLOADS[k]["name"] + ("" if rows is None else f" (first {rows} rows)")
        a_in = qz.amax(x, ws)
        a_out = torch.empty((1,), dtype=torch.float32, device=dev)
        for run in runs:
            fname, gname = run[0], run[1]
            if fname == "asym4":
                out.append({**measure_asym4(name, r, c, run[2], timed, peaks, dev), "workload_id": k})
                continue
            if fname == "qdot":
                out.append({**measure_qdot(name, r, c, run[2], run[3], timed, peaks, dev),
                            "workload_id": k})
                continue
            delayed = len(run) > 2 and run[2] == "delayed"
            bsz = run[2] if len(run) > 2 and isinstance(run[2], int) else None
            f, g = qz.FORMATS[fname], qz.GRANULARITIES[gname]
            codes, scales, ts = qz.alloc_outputs(f, g, r, c, dev, bsz)
            y = torch.empty((r, c), dtype=x.dtype, device=dev)
            d = qz.make_desc(f, idt, g, r, c, block_size=bsz)
            amax_pass = not delayed and (g == qz.QZ_GRAN_TENSOR or
                                         (f == qz.QZ_NVFP4 and g == qz.QZ_GRAN_BLOCK))

            def q(stats_ptr):
                if delayed:
                    rc = qz.qz_quantize_delayed(d, x.data_ptr(), codes.data_ptr(), qz._ptr(scales),
                                                ts.data_ptr(), a_in.data_ptr(), a_out.data_ptr(),
                                                stats_ptr, ws.ptr, sp)
                else:
                    rc = qz.qz_quantize(d, x.data_ptr(), codes.data_ptr(), qz._ptr(scales),
                                        ts.data_ptr(), None, stats_ptr, ws.ptr, sp)
                assert rc == 0, rc

            def dq():
                rc = qz.qz_dequantize(d, codes.data_ptr(), qz._ptr(scales), ts.data_ptr(),
                                      y.data_ptr(), idt, sp)
                assert rc == 0, rc
            qns = timed(lambda: q(None))  # the quantize alone
            qms, dms = timed(lambda: q(st.data_ptr())), timed(dq)
            cb = codes.numel() + (0 if scales is None else scales.numel() * scales.element_size()) + 4
            qb = n * eb * (2 if amax_pass else 1) + cb + 32 + (8 if delayed else 0)
            db = cb + n * eb
            warm = {}
            if k in WARM_WORKLOADS:
                qw, dw = timed(lambda: q(st.data_ptr()), cold=False), timed(dq, cold=False)
                warm = {"quantize_warm_us": round(qw * 1e3, 1),
                        "quantize_warm_frac": round(qb / qw / 1e6 / peaks["hbm_gbs"], 3),
                        "dequantize_warm_us": round(dw * 1e3, 1),
                        "dequantize_warm_frac": round(db / dw / 1e6 / peaks["hbm_gbs"], 3)}
            out.append({"workload": name, "workload_id": k, "format": fname,
                        "granularity": gname + (" delayed" if delayed else "") +
                                       (f" {bsz}" if bsz else ""),
                        "quantize_us": round(qms * 1e3, 1),
                        "quantize_gbs": round(qb / qms / 1e6, 1),
                        "quantize_frac": round(qb / qms / 1e6 / peaks["hbm_gbs"], 3),
                        "quantize_launches": 2 if amax_pass else 1,
                        "quantize_nostats_us": round(qns * 1e3, 1),
                        "quantize_nostats_frac": round(qb / qns / 1e6 / peaks["hbm_gbs"], 3),
                        "dequantize_us": round(dms * 1e3, 1),
                        "dequantize_gbs": round(db / dms / 1e6, 1),
                        "dequantize_frac": round(db / dms / 1e6 / peaks["hbm_gbs"], 3), **warm})
        del x
    if ws.status() != 0:
        raise RuntimeError("status flags set during the format matrix")
    return out


def measure_asym4(name, rows, cols, group, timed, peaks, dev) -> dict:
    """The asymmetric 4-bit group dequantization on a weight of the workload's shape: seeded
    random codes, shifts and scales made on the device (not timed), bf16 output."""
    import torch
    import precision_quantization_gb300 as qz
    gen = torch.Generator(device=dev).manual_seed(7)
    w = torch.randint(-2 ** 31, 2 ** 31 - 1, (rows, cols // 8), dtype=torch.int32, device=dev,
                      generator=gen)
    ng = cols // group
    sc = torch.randn((rows, ng), dtype=torch.float32, device=dev, generator=gen)
    sh = torch.randint(-2 ** 31, 2 ** 31 - 1, (rows, (ng + 7) // 8), dtype=torch.int32,
                       device=dev, generator=gen)
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream

    def dq():
        rc = qz.qz_dequantize_asym4(w.data_ptr(), sc.data_ptr(), sh.data_ptr(), rows, cols, group,
                                    y.data_ptr(), cols, qz.QZ_BF16, sp)
        assert rc == 0, rc
    dms = timed(dq)
    db = w.numel() * 4 + sc.numel() * 4 + sh.numel() * 4 + y.numel() * 2
    return {"workload": name, "format": "asym4", "granularity": f"group {group}",
            "quantize_us": None, "quantize_gbs": None, "quantize_frac": None,
            "quantize_launches": 0,
            "dequantize_us": round(dms * 1e3, 1), "dequantize_gbs": round(db / dms / 1e6, 1),
            "dequantize_frac": round(db / dms / 1e6 / peaks["hbm_gbs"], 3)}


def measure_qdot(name, n0, mid, group, n1, timed, peaks, dev) -> dict:
    """The quantized matrix product z = sum sc (w - sh) y with a weight of the workload's
    shape ([n0, mid], seeded random codes, shifts and scales made on the device) and n1
    bf16 activation columns.  Reported in the dequantize columns: GB/s of weights, scales,
    shifts, activations and outputs moved."""
    import torch
    import precision_quantization_gb300 as qz
    gen = torch.Generator(device=dev).manual_seed(11)
    w = torch.randint(-2 ** 31, 2 ** 31 - 1, (n0, mid // 8), dtype=torch.int32, device=dev,
                      generator=gen)
    ng = mid // group
    sc = torch.randn((n0, ng), dtype=torch.float32, device=dev, generator=gen) * 0.02
    sh = torch.randint(-2 ** 31, 2 ** 31 - 1, (n0, (ng + 7) // 8), dtype=torch.int32,
                       device=dev, generator=gen)
    y = torch.randn((mid, n1), dtype=torch.float32, device=dev, generator=gen).to(torch.bfloat16)
    z = torch.empty((n0, n1), dtype=torch.float32, device=dev)
    sp = torch.cuda.current_stream(dev).cuda_stream

    def run():
        rc = qz.qz_quant_dot(w.data_ptr(), sc.data_ptr(), sh.data_ptr(), n0, mid, group,
                             y.data_ptr(), n1, n1, z.data_ptr(), n1, sp)
        assert rc == 0, rc
    ms = timed(run)
    nb = (w.numel() + sc.numel() + sh.numel()) * 4 + y.numel() * 2 + z.numel() * 4
    row = {"workload": name, "format": "qdot", "granularity": f"group {group} n1 {n1}",
           "quantize_us": None, "quantize_gbs": None, "quantize_frac": None,
           "quantize_launches": 0,
           "dequantize_us": round(ms * 1e3, 1), "dequantize_gbs": round(nb / ms / 1e6, 1),
           "dequantize_frac": round(nb / ms / 1e6 / peaks["hbm_gbs"], 3)}
    if n1 > 8:  # a dense contraction: tensor throughput against the sustained bf16 peak
        tf = 2.0 * n0 * mid * n1 / (ms * 1e-3) / 1e12
        row.update({"tflops": round(tf, 1), "tflops_peak": peaks["bf16_tflops_sustained"],
                    "tflops_frac": round(tf / peaks["bf16_tflops_sustained"], 3),
                    "bound": "tensor", "dtype": "bf16 operands, fp32 accumulation"})
    return row


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def job_gbs(step_bytes: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank processes one full step of the workload (replicas),
    and the job's step time is the slowest rank's."""
    return step_bytes * world / (ms_max * 1e-3) / 1e9


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_baseline(x_np, bytes_per_elem: float, budget_s: float = 12.0, max_rows=None) -> dict:
    """The oracle (as it stands) on a bounded row sample of the same workload, on the host
    cores: MXFP4 and NVFP4 quantize with stats + dequantize to bf16."""
    import oracle as O
    rows = 64
    total_rows = x_np.shape[0] if max_rows is None else min(max_rows, x_np.shape[0])

    def run(r):
        sub = x_np[:r]
        amax = O.amax(x_np)  # global amax of the whole tensor, as the GPU computes it
        t0 = time.perf_counter()
        for fmt in (O.MXFP4, O.NVFP4):
            codes, sc, ts, _ = O.quantize(sub, fmt, O.GRAN_BLOCK,
                                          tensor_amax=amax if fmt == O.NVFP4 else None,
                                          stats=True)
            O.dequantize(codes, sc, ts, fmt, O.GRAN_BLOCK, r, sub.shape[1], out_dtype=O.BF16)
        return time.perf_counter() - t0

    dt = run(rows)
    while dt < budget_s / 4 and rows * 2 <= total_rows:
        rows = min(total_rows, int(rows * max(2.0, min(8.0, budget_s / 2 / max(dt, 1e-3)))))
        dt = run(rows)
    n = rows * x_np.shape[1]
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    gbs = bytes_per_elem * n / dt / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"first {rows} rows x {x_np.shape[1]} of the workload ({n} elements), "
                      f"MXFP4+NVFP4 quantize(+stats)->dequantize, {dt:.2f} s",
            "elements_per_s": round(n / dt, 1), **host_info(), "per_core": oracle_one_thread()}


def host_info() -> dict:
    """CPU model name (lscpu, else /proc/cpuinfo) and machine architecture of the host."""
    import platform
    model = None
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for ln in r.stdout.splitlines():
            if ln.split(":")[0].strip() == "Model name":
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    model = ln.split(":", 1)[1].strip()
                    break
    return {"cpu_model": model, "arch": platform.machine(), "nproc": os.cpu_count()}


def oracle_one_thread() -> dict:
    """The oracle on one thread over the whole small workload (1024 x 1024 bf16, N(0,1)):
    every format of that workload quantized with statistics and dequantized to bf16 --
    the per-core rate of the CPU baseline."""
    import oracle as O
    import workloads as W
    x = W.workload(1)
    n = x.size
    runs = [(O.INT8, O.GRAN_TENSOR), (O.E4M3, O.GRAN_TENSOR), (O.MXFP4, O.GRAN_BLOCK),
            (O.NVFP4, O.GRAN_BLOCK)]
    nbytes = 0
    t0 = time.perf_counter()
    for fmt, gran in runs:
        codes, sc, ts, _ = O.quantize(x, fmt, gran, stats=True, nthreads=1)
        O.dequantize(codes, sc, ts, fmt, gran, x.shape[0], x.shape[1], out_dtype=O.BF16,
                     nthreads=1)
        out = codes.nbytes + (0 if sc is None else sc.nbytes) + 4
        nbytes += 2 * (2 * n + out)  # quantize: x in, codes out; dequantize: codes in, y out
    dt = time.perf_counter() - t0
    return {"threads": 1, "workload": "normal-1024x1024-bf16",
            "ops": "INT8, E4M3 (tensor), MXFP4, NVFP4: quantize(+stats) -> dequantize(bf16)",
            "seconds": round(dt, 3), "gbs": round(nbytes / dt / 1e9, 4),
            "elements_per_s": round(len(runs) * n / dt, 1)}


def run_reference(args, world, rank):
    """The CPU oracle timed as the reference arm, on bounded samples of the workload."""
    if rank != 0:
        return
    import numpy as np
    import workloads as W
    import oracle as O
    x = W.workload(4)
    n = ROWS * COLS
    bpe = sum(algorithmic_bytes(n).values()) / n
    sample_rows = 256
    amax = O.amax(x)

    def step():
        sub = x[:sample_rows]
        for fmt in (O.MXFP4, O.NVFP4):
            codes, sc, ts, _ = O.quantize(sub, fmt, O.GRAN_BLOCK,
                                          tensor_amax=amax if fmt == O.NVFP4 else None,
                                          stats=True)
            O.dequantize(codes, sc, ts, fmt, O.GRAN_BLOCK, sample_rows, COLS, out_dtype=O.BF16)

    for _ in range(args.warmup):
        step()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    dt = statistics.mean(times)
    ne = sample_rows * COLS
    value = bpe * ne / dt / 1e9
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "rows": ROWS, "cols": COLS,
                   "formats": ["mxfp4", "nvfp4"], "sample_rows_per_step": sample_rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": f"first {sample_rows} rows x {COLS} per step ({ne} elements)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "elements_per_s": round(ne / dt, 1),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--e2e-chunk-rows", type=int, default=4096,
                    help="rows per host-to-device copy of the end-to-end round trip")
    ap.add_argument("--no-matrix", action="store_true",
                    help="skip the per-format matrix over the five workloads")
    ap.add_argument("--matrix-only", action="store_true",
                    help="print only the per-format matrix (one JSON line)")
    ap.add_argument("--matrix-workloads", default="1,2,3,4,5",
                    help="comma-separated workload numbers of the matrix")
    ap.add_argument("--qdot-sweep", action="store_true",
                    help="print only the quantized-product sweep (one JSON line, TFLOP/s)")
    ap.add_argument("--matrix-rows", type=int, default=None,
                    help="at most this many rows of each matrix workload (small cases for profiling)")
    ap.add_argument("--rows", type=int, default=ROWS,
                    help="rows of the workload (same recipe); the default is the full size")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()

    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    import numpy as np
    import torch
    import precision_quantization_gb300 as qz
    import workloads as W

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    which = tuple(int(v) for v in args.matrix_workloads.split(",") if v)
    if args.qdot_sweep:
        flush = L2Flush(dev)
        m = measure_qdot_sweep(dev, measured_peaks(), flush)
        print(json.dumps({"metric": "quantized product TFLOP/s (bf16 tensor cores)", "unit": "TFLOP/s",
                          "products": m}), flush=True)
        return
    if args.matrix_only:
        flush = L2Flush(dev)
        m = measure_matrix(dev, measured_peaks(), flush, which=which, max_rows=args.matrix_rows)
        print(json.dumps({"metric": METRIC, "unit": "GB/s", "formats": m}), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    rows = args.rows
    x_np = W.workload(4, rows=rows)
    n = rows * COLS
    x = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).to(dev)
    ws = qz.Workspace(dev)
    outs = {f: qz.alloc_outputs(f, qz.QZ_GRAN_BLOCK, rows, COLS, dev)
            for f in (qz.QZ_MXFP4, qz.QZ_NVFP4)}
    ys = {f: torch.empty((rows, COLS), dtype=torch.bfloat16, device=dev) for f in outs}
    sts = {f: torch.empty((qz.STATS_BYTES,), dtype=torch.uint8, device=dev) for f in outs}
    amax_buf = torch.empty((1,), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    desc = {f: qz.make_desc(f, qz.QZ_BF16, qz.QZ_GRAN_BLOCK, rows, COLS) for f in outs}
    desc_amax = qz.make_desc(qz.QZ_INT8, qz.QZ_BF16, qz.QZ_GRAN_TENSOR, rows, COLS)
    names = ["mx_quant", "mx_dequant", "nv_amax", "nv_quant", "nv_dequant"]
    abytes = algorithmic_bytes(n)
    step_bytes = sum(abytes.values())

    def launches(x_ptr, ev=None):
        """The 5 launches of one step; ev: optional list of 6 events bracketing them."""
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        c, s, t = outs[qz.QZ_MXFP4]
        rc = qz.qz_quantize(desc[qz.QZ_MXFP4], x_ptr, c.data_ptr(), s.data_ptr(), t.data_ptr(),
                            None, sts[qz.QZ_MXFP4].data_ptr(), ws.ptr, sptr)
        mark(1)
        rc |= qz.qz_dequantize(desc[qz.QZ_MXFP4], c.data_ptr(), s.data_ptr(), t.data_ptr(),
                               ys[qz.QZ_MXFP4].data_ptr(), qz.QZ_BF16, sptr)
        mark(2)
        rc |= qz.qz_amax(desc_amax, x_ptr, amax_buf.data_ptr(), ws.ptr, sptr)
        mark(3)
        c, s, t = outs[qz.QZ_NVFP4]
        rc |= qz.qz_quantize(desc[qz.QZ_NVFP4], x_ptr, c.data_ptr(), s.data_ptr(), t.data_ptr(),
                             amax_buf.data_ptr(), sts[qz.QZ_NVFP4].data_ptr(), ws.ptr, sptr)
        mark(4)
        rc |= qz.qz_dequantize(desc[qz.QZ_NVFP4], c.data_ptr(), s.data_ptr(), t.data_ptr(),
                               ys[qz.QZ_NVFP4].data_ptr(), qz.QZ_BF16, sptr)
        mark(5)
        if rc != 0:
            raise RuntimeError(f"libqz call failed ({rc})")

    clk = ClockSampler(local).__enter__()
    for _ in range(args.warmup):
        flush.run()
        launches(x.data_ptr())
    torch.cuda.synchronize(dev)
    if ws.status() != 0:
        raise RuntimeError("non-finite input flagged")
    clk.wait_first()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for k in range(args.steps):
        flush.run()  # L2 flush between timed steps (outside the events)
        launches(x.data_ptr(), evs[k])
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    clk.window(t0, t0 + wall)
    clk.__exit__()
    if world > 1:
        torch.distributed.barrier()
    per_kernel = {nm: [] for nm in names}
    step_ms = []
    for ev in evs:
        step_ms.append(ev[0].elapsed_time(ev[5]))
        for i, nm in enumerate(names):
            per_kernel[nm].append(ev[i].elapsed_time(ev[i + 1]))
    ms = statistics.mean(step_ms)
    ms = max_over_ranks(ms, world, dev)
    value = job_gbs(step_bytes, world, ms)
    peaks = measured_peaks()
    kern = {}
    for nm in names:
        avg = statistics.mean(per_kernel[nm])
        kern[nm] = {"ms": round(avg, 5), "gbs": round(abytes[nm] / (avg * 1e-3) / 1e9, 1),
                    "frac_hbm": round(abytes[nm] / (avg * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
    dominant = max(names, key=lambda nm: kern[nm]["ms"])
    achieved = abytes[dominant] / (kern[dominant]["ms"] * 1e-3) / 1e9
    stats_host = {f: qz.read_stats(sts[f]) for f in outs}

    # ---- end to end through the public API: pinned host input in, quantized tensors out
    e2e = None
    if not args.no_e2e:
        from precision_quantization_gb300.streamed import HostRoundTrip
        xh = torch.from_numpy(x_np.view(np.int16)).view(torch.bfloat16).pin_memory()
        # the same five operations as the kernel step, on row chunks as they arrive
        plan = HostRoundTrip(rows, COLS, [(qz.QZ_MXFP4, qz.QZ_GRAN_BLOCK),
                                          (qz.QZ_NVFP4, qz.QZ_GRAN_BLOCK)],
                             chunk_rows=args.e2e_chunk_rows, device=dev)
        h2d = plan.bytes_in()
        d2h = plan.bytes_out()
        for _ in range(max(3, args.warmup)):
            plan.run(xh)
        e_ms = []
        for _ in range(args.e2e_steps):
            flush.run()
            torch.cuda.synchronize(dev)
            t1 = time.perf_counter()
            plan.run(xh)
            e_ms.append((time.perf_counter() - t1) * 1e3)
        if plan.status() != 0:
            raise RuntimeError("e2e: device status flags raised")
        for j, f in enumerate((qz.QZ_MXFP4, qz.QZ_NVFP4)):  # same statistics as the kernel step
            a, b = plan.read_stats(j), stats_host[f]
            if a.n != b.n or a.max_abs_err != b.max_abs_err or a.max_rel_err != b.max_rel_err \
                    or abs(a.sum_sq_err - b.sum_sq_err) > 1e-5 * abs(b.sum_sq_err):
                raise RuntimeError(f"e2e statistics differ from the kernel step's: {a} {b}")
        # median: a host clock around each round trip sees the odd scheduling hiccup of the
        # host thread (tens of ms), which would dominate a mean over a few steps
        em = max_over_ranks(statistics.median(e_ms), world, dev)
        e2e = {"value": round(job_gbs(step_bytes, world, em), 2), "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(em, 3), "ms_mean": round(statistics.mean(e_ms), 3),
               "steps": len(e_ms), "timing": "host clock per round trip, median",
               "chunk_rows": args.e2e_chunk_rows,
               "api": "qz_host_run, one C-ABI call per round trip (pinned host in/out, "
                      "copies overlapped with the kernels on the library's own streams)"}

    matrix = None
    if not args.no_matrix and rank == 0:
        matrix = measure_matrix(dev, measured_peaks(), flush, x4=x if rows == ROWS else None,
                                which=which)
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(x_np, step_bytes / n)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD if rows == ROWS else f"{WORKLOAD} (first {rows} rows)",
                   "rows": rows, "cols": COLS, "input": "bf16",
                   "formats": ["mxfp4", "nvfp4"],
                   "step": "mx quantize(+stats)->dequantize(bf16); nv amax->quantize(+stats)"
                           "->dequantize(bf16)",
                   "bytes_per_step": step_bytes,
                   "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write, then "
                         f"{L2_FLUSH_BYTES >> 20} MiB read to write its dirty lines back); "
                         "input 512 MiB > L2",
                   "parallelism": f"replicas x{world}"},
        "elements_per_s": round(n * 2 * world / (ms * 1e-3), 1),
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4),
                     "peak_source": peaks["source"], "traffic": recorded_traffic(dominant),
                     "algorithmic_bytes_per_launch": abytes[dominant]},
        "kernels": kern,
        "per_format": {
            "mxfp4": {"round_trip_gbs": round((abytes["mx_quant"] + abytes["mx_dequant"]) /
                      ((kern["mx_quant"]["ms"] + kern["mx_dequant"]["ms"]) * 1e-3) / 1e9, 1),
                      "mse": stats_host[qz.QZ_MXFP4].mse,
                      "max_rel_err": stats_host[qz.QZ_MXFP4].max_rel_err},
            "nvfp4": {"round_trip_gbs": round((abytes["nv_amax"] + abytes["nv_quant"] +
                      abytes["nv_dequant"]) / ((kern["nv_amax"]["ms"] + kern["nv_quant"]["ms"] +
                      kern["nv_dequant"]["ms"]) * 1e-3) / 1e9, 1),
                      "mse": stats_host[qz.QZ_NVFP4].mse,
                      "max_rel_err": stats_host[qz.QZ_NVFP4].max_rel_err},
        },
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * len(names),
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 4),
    }
    # the verbose matrix first and the compact one last: a reader that keeps only the end
    # of the line still has every per-format cell
    line = {"formats": matrix, **line}
    line["format_fracs"] = None if matrix is None else compact_matrix(matrix)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
