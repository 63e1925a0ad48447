"""GPU parity of the chunked host round trip (HostRoundTrip) and of qz_stats_merge.

The round trip copies x from pinned host memory in row chunks and quantizes each chunk
as it lands (per-tensor scales after every chunk is in); its codes, scales, tensor scale
and dequantized values must equal the oracle's quantization of the whole tensor bit for
bit, and its merged statistics must match the oracle's as the fused statistics do."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import assert_stats_close, run_oracle, to_device, to_host_bits, torch_mod

pytestmark = pytest.mark.gpu


def host_tensor(x_np):
    torch = torch_mod()
    if x_np.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x_np))
    return t.pin_memory()


def check_run(plan, j, x_np, fmt, gran):
    import precision_quantization_gb300 as qz
    out_dt = "bf16" if plan.out_code == qz.QZ_BF16 else "f32"
    o = run_oracle(x_np, fmt, gran, out_dtypes=(out_dt,))
    h = plan.host[j]
    assert np.array_equal(h["codes"].numpy(), o["codes"]), (fmt, gran, "codes")
    if o["scales"] is not None:
        s = h["scales"].numpy()
        s = s.view(np.uint32) if s.dtype == np.float32 else s
        assert np.array_equal(s, o["scales"]), (fmt, gran, "scales")
    if gran != O.GRAN_ROW and not (fmt == O.MXFP4 and gran == O.GRAN_BLOCK):
        assert h["tensor_scale"].numpy().view(np.uint32)[0] == np.float32(o["ts"]).view(np.uint32)
    assert np.array_equal(to_host_bits(plan.y[j]), o["y"][out_dt]), (fmt, gran, "dequantized")
    assert_stats_close(plan.read_stats(j), o["stats"], f"merged {fmt} {gran}")


RUNS = [(O.MXFP4, O.GRAN_BLOCK), (O.NVFP4, O.GRAN_BLOCK), (O.E4M3, O.GRAN_TENSOR),
        (O.INT8, O.GRAN_ROW)]


@pytest.mark.parametrize("chunk_rows", [384, 1000, 4096, 1])
def test_round_trip_lognormal_chunks(chunk_rows):
    """Workload-4-like rows (log-normal magnitudes), ragged last chunk, one-row chunks, and
    a chunk larger than the tensor."""
    from precision_quantization_gb300.streamed import HostRoundTrip
    rows, cols = (1000, 512) if chunk_rows > 1 else (37, 256)
    x_np = W.lognormal_signed(rows, cols, seed=41)
    plan = HostRoundTrip(rows, cols, RUNS, chunk_rows=chunk_rows)
    plan.run(host_tensor(x_np))
    for j, (f, g) in enumerate(RUNS):
        check_run(plan, j, x_np, f, g)
    assert plan.status() == 0


def test_round_trip_reused_plan_f32_edge_mix():
    """fp32 edge-case input (ties, subnormals, saturation, signed zeros); the plan is run on
    two different tensors in a row and must give each one's own results."""
    from precision_quantization_gb300.streamed import HostRoundTrip
    runs = [(O.NVFP4, O.GRAN_BLOCK), (O.E5M2, O.GRAN_TENSOR), (O.MXFP4, O.GRAN_BLOCK),
            (O.INT8, O.GRAN_UNIT)]
    rows, cols = 300, 256
    plan = HostRoundTrip(rows, cols, runs, in_dtype="f32", chunk_rows=128, out_dtype="f32")
    for seed in (51, 52):
        x_np = W.edge_mix(rows, cols, seed=seed)
        plan.run(host_tensor(x_np))
        for j, (f, g) in enumerate(runs):
            check_run(plan, j, x_np, f, g)


def test_round_trip_without_stats():
    """The plan without the fused statistics: the same codes, scales and dequantized values
    (the NVFP4 and TENSOR formats still take their amax over all chunks)."""
    from precision_quantization_gb300.streamed import HostRoundTrip
    rows, cols = 513, 1024
    x_np = W.activation_like(rows, cols, seed=71)
    plan = HostRoundTrip(rows, cols, RUNS, chunk_rows=200, stats=False)
    plan.run(host_tensor(x_np))
    for j, (f, g) in enumerate(RUNS):
        o = run_oracle(x_np, f, g, stats=False, out_dtypes=("bf16",))
        h = plan.host[j]
        assert np.array_equal(h["codes"].numpy(), o["codes"]), (f, g)
        if o["scales"] is not None:
            sc = h["scales"].numpy()
            assert np.array_equal(sc.view(np.uint32) if sc.dtype == np.float32 else sc, o["scales"])
        assert np.array_equal(to_host_bits(plan.y[j]), o["y"]["bf16"]), (f, g)
    assert plan.bytes_out() == sum(t.numel() * t.element_size() for h in plan.host
                                   for k, t in h.items() if t is not None and k != "stats")


def test_round_trip_int4_unit_and_row_scales():
    """Scale layouts the other cases leave out: INT4 groups of 32 (fp32 scales per group),
    MXFP4 and NVFP4 UNIT (scale bytes of value 1 per block), E5M2 ROW; fp32 input and f32
    dequantized outputs, a ragged last chunk."""
    from precision_quantization_gb300.streamed import HostRoundTrip
    runs = [(O.INT4, O.GRAN_BLOCK), (O.MXFP4, O.GRAN_UNIT), (O.NVFP4, O.GRAN_UNIT), (O.E5M2, O.GRAN_ROW)]
    rows, cols = 203, 512
    x_np = W.lognormal_signed(rows, cols, seed=45, dtype="f32")
    plan = HostRoundTrip(rows, cols, runs, in_dtype="f32", chunk_rows=64, out_dtype="f32")
    plan.run(host_tensor(x_np))
    for j, (f, g) in enumerate(runs):
        check_run(plan, j, x_np, f, g)
    assert plan.status() == 0


def test_round_trip_pageable_input():
    """A host tensor that is not page-locked: the copies do not overlap, the results are
    the same."""
    from precision_quantization_gb300.streamed import HostRoundTrip
    torch = torch_mod()
    rows, cols = 257, 512
    x_np = W.lognormal_signed(rows, cols, seed=43)
    xh = torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).view(torch.bfloat16)
    assert not xh.is_pinned()
    plan = HostRoundTrip(rows, cols, RUNS, chunk_rows=100)
    plan.run(xh)
    for j, (f, g) in enumerate(RUNS):
        check_run(plan, j, x_np, f, g)


def test_host_run_missing_buffer():
    """A required device buffer missing from one run's io: QZ_ERR_NULL before anything is
    enqueued, and the plan still works afterwards."""
    import precision_quantization_gb300 as qz
    from precision_quantization_gb300.streamed import HostRoundTrip
    rows, cols = 64, 256
    x_np = W.activation_like(rows, cols, seed=44)
    plan = HostRoundTrip(rows, cols, RUNS, chunk_rows=32)
    xh = host_tensor(x_np)
    for field in ("codes", "scales", "tensor_scale", "stats"):
        io = [qz.QzHostIo.from_buffer_copy(v) for v in plan.io]
        j = 0 if field == "scales" else 2  # MXFP4 has scales; E4M3 TENSOR has none
        setattr(io[j], field, None)
        assert qz.qz_host_run(plan.plan, xh.data_ptr(), io) == qz.QZ_ERR_NULL, field
    assert qz.qz_host_run(plan.plan, None, plan.io) == qz.QZ_ERR_NULL  # x_host
    plan.run(xh)
    for j, (f, g) in enumerate(RUNS):
        check_run(plan, j, x_np, f, g)
    assert plan.status() == 0


def test_round_trip_empty():
    from precision_quantization_gb300.streamed import HostRoundTrip
    torch = torch_mod()
    plan = HostRoundTrip(0, 64, [(O.NVFP4, O.GRAN_BLOCK), (O.MXFP4, O.GRAN_BLOCK)])
    plan.run(torch.empty((0, 64), dtype=torch.bfloat16).pin_memory())
    for j in range(2):
        s = plan.read_stats(j)
        assert s.n == 0 and s.sum_sq_err == 0 and s.mse == 0


@pytest.mark.parametrize("fmt,gran", [(O.NVFP4, O.GRAN_BLOCK), (O.E4M3, O.GRAN_ROW),
                                      (O.MXFP4, O.GRAN_BLOCK)])
def test_stats_merge_of_row_parts(fmt, gran):
    """Statistics of three row ranges (one of a single row), each quantized with the
    whole tensor's amax, merged: equal to the oracle's statistics of the whole tensor.  The
    merge may write over its first part."""
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    rows, cols = 301, 256
    x_np = W.activation_like(rows, cols, seed=61)
    x = to_device(x_np)
    alpha = torch.tensor([float(O.amax(x_np))], dtype=torch.float32, device=x.device)
    ws = qz.Workspace(x.device)
    cuts = [(0, 120), (120, 121), (121, rows)]
    parts = torch.empty((len(cuts), qz.STATS_BYTES), dtype=torch.uint8, device=x.device)
    needs_alpha = fmt == O.NVFP4 or gran == O.GRAN_TENSOR
    for i, (r0, r1) in enumerate(cuts):
        q, st = qz.quantize(x[r0:r1], fmt, gran, tensor_amax=alpha if needs_alpha else None,
                            stats=True, workspace=ws)
        parts[i].copy_(st)
    merged = torch.empty((qz.STATS_BYTES,), dtype=torch.uint8, device=x.device)
    assert qz.qz_stats_merge(parts.data_ptr(), len(cuts), merged.data_ptr(), 0) == qz.QZ_OK
    assert qz.qz_stats_merge(parts.data_ptr(), len(cuts), parts[0].data_ptr(), 0) == qz.QZ_OK
    torch.cuda.synchronize()
    alpha_o = np.float32(O.amax(x_np)) if needs_alpha else None
    _, _, _, st_o = O.quantize(x_np, fmt, gran, O.SCALE_UP, alpha_o, True)
    assert_stats_close(qz.read_stats(merged), st_o, "merged")
    assert_stats_close(qz.read_stats(parts[0]), st_o, "merged in place")


def test_stats_merge_arguments():
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    out = torch.full((qz.STATS_BYTES,), 7, dtype=torch.uint8, device="cuda")
    assert qz.qz_stats_merge(None, 0, out.data_ptr(), 0) == qz.QZ_OK
    torch.cuda.synchronize()
    s = qz.read_stats(out)
    assert (s.n, s.sum_sq_err, s.mse, s.max_abs_err, s.max_rel_err) == (0, 0.0, 0.0, 0.0, 0.0)
    assert qz.qz_stats_merge(out.data_ptr(), -1, out.data_ptr(), 0) == qz.QZ_ERR_SHAPE
    assert qz.qz_stats_merge(None, 2, out.data_ptr(), 0) == qz.QZ_ERR_NULL
    assert qz.qz_stats_merge(out.data_ptr(), 1, None, 0) == qz.QZ_ERR_NULL
    assert qz.qz_stats_merge(out.data_ptr() + 4, 1, out.data_ptr(), 0) == qz.QZ_ERR_ALIGN
