"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, element by element.

Codes, scales, tensor scales and dequantized values (bf16 and fp32) must be bit-exact;
max |e|, max |e|/|x| and n bit-exact; the sum of squares and MSE within 1e-5 relative.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import assert_parity, run_gpu, run_oracle, to_device, torch_mod

pytestmark = pytest.mark.gpu

FMT8 = [O.INT8, O.E4M3, O.E5M2]
FMT4 = [O.MXFP4, O.NVFP4]


def gen(rows, cols, dtype, seed, kind="lognormal"):
    if kind == "lognormal":
        x = W.lognormal_signed(rows, cols, seed=seed, sigma=2.0, dtype="f32")
    elif kind == "edge":
        x = W.edge_mix(rows, cols, seed=seed)
    else:
        x = W.normal(rows, cols, 1.0, seed=seed, dtype="f32")
    return W.bf16_bits(x) if dtype == "bf16" else x


SHAPES8 = [(1, 16), (2, 7), (3, 48), (5, 1000), (33, 64), (257, 1024), (64, 4096), (4, 33)]
SHAPES4 = [(1, 32), (3, 64), (33, 96), (257, 1024), (64, 4096), (7, 160)]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("gran", [O.GRAN_TENSOR, O.GRAN_ROW, O.GRAN_UNIT])
@pytest.mark.parametrize("fmt", FMT8)
def test_parity_8bit(fmt, gran, dtype):
    for i, (r, c) in enumerate(SHAPES8):
        kind = "edge" if (dtype == "f32" and i % 2) else "lognormal"
        x = gen(r, c, dtype, seed=100 + i, kind=kind)
        assert_parity(run_gpu(x, fmt, gran), run_oracle(x, fmt, gran))


@pytest.mark.parametrize("scale_round", [O.SCALE_UP, O.SCALE_NEAREST])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("gran", [O.GRAN_BLOCK, O.GRAN_UNIT])
@pytest.mark.parametrize("fmt", FMT4)
def test_parity_fp4(fmt, gran, dtype, scale_round):
    for i, (r, c) in enumerate(SHAPES4):
        kind = "edge" if (dtype == "f32" and i % 2) else "lognormal"
        x = gen(r, c, dtype, seed=200 + i, kind=kind)
        assert_parity(run_gpu(x, fmt, gran, scale_round),
                      run_oracle(x, fmt, gran, scale_round))


@pytest.mark.parametrize("fmt,gran", [(O.INT8, O.GRAN_ROW), (O.E4M3, O.GRAN_TENSOR),
                                      (O.E5M2, O.GRAN_UNIT), (O.MXFP4, O.GRAN_BLOCK),
                                      (O.NVFP4, O.GRAN_BLOCK)])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("pad", [1, 8, 37])
def test_parity_strided_rows(fmt, gran, dtype, pad):
    """x as a view with leading dimension cols + pad (element-wise and vector paths)."""
    x = gen(19, 128, dtype, seed=300 + pad)
    assert_parity(run_gpu(x, fmt, gran, ld_pad=pad), run_oracle(x, fmt, gran))


@pytest.mark.parametrize("kind", ["lognormal", "edge"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("fmt", FMT8)
def test_parity_row_without_stats(fmt, dtype, kind):
    """Per-row scales without the fused statistics (short rows take a kernel of their
    own there: a warp per row, 2 / 4 / 8 chunks per lane), including rows of one chunk,
    ragged widths and rows too long for it."""
    for i, (rows, cols) in enumerate(SHAPES8 + [(300, 2048), (1000, 512), (77, 4096 + 16)]):
        x = gen(rows, cols, dtype, seed=700 + i, kind=kind)
        assert_parity(run_gpu(x, fmt, O.GRAN_ROW, stats=False),
                      run_oracle(x, fmt, O.GRAN_ROW, stats=False), stats=False)


@pytest.mark.parametrize("fmt,gran", [(O.INT8, O.GRAN_TENSOR), (O.E4M3, O.GRAN_TENSOR),
                                      (O.E5M2, O.GRAN_TENSOR), (O.NVFP4, O.GRAN_BLOCK)])
@pytest.mark.parametrize("factor", [1.0, 0.25, 4.0, 1e-30, 0.0])
def test_supplied_tensor_amax(fmt, gran, factor):
    """The per-tensor alpha / NVFP4 global amax given by the caller, equal to, below (values
    saturate), or above the true amax; 0 means unit scale."""
    x = gen(40, 256, "bf16", seed=400)
    a = np.float32(float(O.amax(x)) * factor)
    assert_parity(run_gpu(x, fmt, gran, tensor_amax=a), run_oracle(x, fmt, gran, tensor_amax=a))


@pytest.mark.parametrize("fmt", FMT8 + FMT4)
def test_element_cast_sweep(fmt):
    """Unit scale: the element cast on a sweep of fp32 bit patterns across every binade
    from fp32 denormals to 2^40, both signs, plus the exact midpoints of the grid."""
    bits = []
    for e in range(0, 168):
        bits.append((e << 23) + np.arange(0, 1 << 23, 4099, dtype=np.uint32))
    b = np.concatenate(bits).astype(np.uint32)
    b = np.concatenate([b, b | np.uint32(0x80000000)])
    cols = 64
    b = np.concatenate([b, np.zeros((-len(b)) % cols, dtype=np.uint32)])
    x = b.view(np.float32).reshape(-1, cols)
    assert_parity(run_gpu(x, fmt, O.GRAN_UNIT, out_dtypes=("f32",)),
                  run_oracle(x, fmt, O.GRAN_UNIT, out_dtypes=("f32",)))


@pytest.mark.parametrize("fmt", FMT8)
def test_relative_error_without_zero_codes(fmt):
    """No element rounds to zero, so max |e|/|x| < 1 and the exact-maximum search has to
    find it among ordinary elements."""
    rng = np.random.default_rng(500)
    x = (rng.uniform(0.55, 1.0, (300, 512)) * rng.choice([-1, 1], (300, 512))).astype(np.float32)
    for gran in (O.GRAN_TENSOR, O.GRAN_ROW):
        g, o = run_gpu(x, fmt, gran), run_oracle(x, fmt, gran)
        assert o["stats"].max_rel_err < 1
        assert_parity(g, o)


@pytest.mark.parametrize("fmt,gran", [(O.INT8, O.GRAN_TENSOR), (O.E4M3, O.GRAN_ROW),
                                      (O.MXFP4, O.GRAN_BLOCK), (O.NVFP4, O.GRAN_BLOCK),
                                      (O.NVFP4, O.GRAN_UNIT)])
def test_zero_and_signed_zero(fmt, gran):
    x = np.zeros((5, 64), dtype=np.float32)
    x[1] = -0.0
    x[2, 5] = -0.0
    assert_parity(run_gpu(x, fmt, gran), run_oracle(x, fmt, gran))
    x[3, :] = np.float32(-1e-42)  # denormals in an otherwise zero tensor
    assert_parity(run_gpu(x, fmt, gran), run_oracle(x, fmt, gran))


@pytest.mark.parametrize("fmt,gran", [(O.E4M3, O.GRAN_TENSOR), (O.INT8, O.GRAN_ROW),
                                      (O.NVFP4, O.GRAN_BLOCK), (O.MXFP4, O.GRAN_BLOCK)])
def test_tiny_and_huge_tensors(fmt, gran):
    """Scales far outside the range of the FMA-corrected quotient (IEEE division path)."""
    rng = np.random.default_rng(600)
    for scale in (1e-40, 1e-35, 1e-25, 1e25, 3e36):
        x = (rng.standard_normal((6, 64)) * scale).astype(np.float32)
        assert_parity(run_gpu(x, fmt, gran), run_oracle(x, fmt, gran))


@pytest.mark.parametrize("scale_round", [O.SCALE_UP, O.SCALE_NEAREST])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("fmt", FMT4)
def test_rows_of_mixed_magnitude(fmt, dtype, scale_round):
    """Rows scaled by 10^u, u uniform in [-35, 32]: the chunks' squared errors leave the
    plain fp32 range in some rows and not in others (range buckets of the fused sum), and
    the MXFP4 exponent comes from both the amax-field rule and the division route."""
    rng = np.random.default_rng(610)
    x = W.lognormal_signed(96, 4096, seed=611, sigma=2.0, dtype="f32")
    x = (x * (10.0 ** rng.uniform(-35, 32, size=(96, 1)))).astype(np.float32)
    x[5] = 0.0
    x[7, :64] = np.float32(3e-41)
    if dtype == "bf16":
        x = W.bf16_bits(x)
    assert_parity(run_gpu(x, fmt, O.GRAN_BLOCK, scale_round=scale_round),
                  run_oracle(x, fmt, O.GRAN_BLOCK, scale_round=scale_round))


@pytest.mark.parametrize("fmt,gran", [(O.E5M2, O.GRAN_TENSOR), (O.INT8, O.GRAN_ROW),
                                      (O.MXFP4, O.GRAN_BLOCK), (O.NVFP4, O.GRAN_BLOCK)])
def test_empty(fmt, gran):
    import precision_quantization_gb300 as qz
    import torch
    for r, c in ((0, 64), (3, 0), (0, 0)):
        x = torch.zeros((r, c), dtype=torch.bfloat16, device="cuda")
        q, st = qz.quantize(x, fmt, gran, stats=True)
        y = qz.dequantize(q)
        torch.cuda.synchronize()
        s = qz.read_stats(st)
        assert s.n == 0 and s.mse == 0 and s.sum_sq_err == 0 and y.shape == (r, c)


def test_nonfinite_input_sets_status():
    import precision_quantization_gb300 as qz
    import torch
    x = torch.ones((8, 64), dtype=torch.float32, device="cuda")
    x[3, 7] = float("nan")
    x[5, 9] = float("inf")
    for fmt, gran in ((qz.QZ_NVFP4, "block"), (qz.QZ_MXFP4, "block"), (qz.QZ_INT8, "tensor"),
                      (qz.QZ_FP8_E4M3, "row"), (qz.QZ_FP8_E5M2, "unit")):
        ws = qz.Workspace()
        qz.quantize(x, fmt, gran, stats=True, workspace=ws)
        assert ws.status() & qz.QZ_FLAG_NONFINITE_INPUT, (fmt, gran)
        ws.clear()
        assert ws.status() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("bad", [float("nan"), float("inf"), float("-inf")])
@pytest.mark.parametrize("fmt,gran,sr", [(O.NVFP4, O.GRAN_BLOCK, O.SCALE_UP),
                                         (O.NVFP4, O.GRAN_BLOCK, O.SCALE_NEAREST),
                                         (O.MXFP4, O.GRAN_BLOCK, O.SCALE_UP),
                                         (O.MXFP4, O.GRAN_BLOCK, O.SCALE_NEAREST),
                                         (O.NVFP4, O.GRAN_UNIT, O.SCALE_UP),
                                         (O.MXFP4, O.GRAN_UNIT, O.SCALE_UP)])
def test_fp4_quantize_flags_nonfinite_itself(fmt, gran, sr, bad, dtype):
    """One NaN or +-Inf element, the NVFP4 tensor amax supplied (finite), so no amax pass
    runs: the FP4 quantize kernel must raise the flag itself, with and without the fused
    statistics, and on the delayed path."""
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    x = torch.ones((64, 256), dtype=torch.float32, device="cuda")
    x[17, 100] = bad
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    alpha = torch.ones((1,), dtype=torch.float32, device="cuda")
    ta = alpha if (fmt == O.NVFP4 and gran == O.GRAN_BLOCK) else None
    for stats in (True, False):
        ws = qz.Workspace()
        qz.quantize(x, fmt, gran, sr, tensor_amax=ta, stats=stats, workspace=ws)
        assert ws.status() & qz.QZ_FLAG_NONFINITE_INPUT, (fmt, gran, sr, bad, stats)
    ws = qz.Workspace()
    qz.quantize_delayed(x, fmt, ta, gran, sr, stats=True, workspace=ws)
    assert ws.status() & qz.QZ_FLAG_NONFINITE_INPUT, (fmt, gran, sr, bad, "delayed")


def test_bad_supplied_amax_sets_status():
    import precision_quantization_gb300 as qz
    import torch
    x = torch.ones((8, 64), dtype=torch.bfloat16, device="cuda")
    ws = qz.Workspace()
    bad = torch.tensor([-1.0], device="cuda")
    qz.quantize(x, qz.QZ_FP8_E4M3, "tensor", tensor_amax=bad, workspace=ws, stats=True)
    assert ws.status() & qz.QZ_FLAG_BAD_AMAX


@pytest.mark.parametrize("fmt,gran", [(O.INT8, O.GRAN_ROW), (O.E4M3, O.GRAN_TENSOR),
                                      (O.MXFP4, O.GRAN_BLOCK), (O.NVFP4, O.GRAN_BLOCK)])
def test_guard_bands(fmt, gran):
    """Outputs written into the middle of canary-filled buffers: nothing outside the
    output ranges changes (odd row count, ragged for the 8-bit formats)."""
    import precision_quantization_gb300 as qz
    import torch
    rows, cols = 37, (96 if fmt in FMT4 else 100)
    x_np = gen(rows, cols, "bf16", seed=700)
    x = to_device(x_np)
    G = 4096
    codes_n = rows * cols // (2 if fmt in FMT4 else 1)
    cbuf = torch.full((codes_n + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
    codes = cbuf[G:G + codes_n].view(rows, -1)
    if fmt in FMT4:
        sn = rows * cols // (32 if fmt == O.MXFP4 else 16)
        sbuf = torch.full((sn + 2 * G,), 0x5A, dtype=torch.uint8, device="cuda")
        scales = sbuf[G:G + sn].view(rows, -1)
    else:
        sn = rows
        sbuf = torch.full((sn + 2 * G,), -7.0, dtype=torch.float32, device="cuda")
        scales = sbuf[G:G + sn] if gran == O.GRAN_ROW else None
    tsb = torch.full((8,), -3.0, dtype=torch.float32, device="cuda")
    q, _ = qz.quantize(x, fmt, gran, out=(codes, scales, tsb[4:5]), stats=True)
    ybuf = torch.full((rows * cols + 2 * G,), -5.0, dtype=torch.float32, device="cuda")
    qz.dequantize(q, torch.float32, out=ybuf[G:G + rows * cols].view(rows, cols))
    torch.cuda.synchronize()
    cb = cbuf.cpu().numpy()
    assert (cb[:G] == 0xA5).all() and (cb[-G:] == 0xA5).all()
    sb = sbuf.cpu().numpy()
    if fmt in FMT4:
        assert (sb[:G] == 0x5A).all() and (sb[-G:] == 0x5A).all()
    else:
        assert (sb[:G] == -7).all() and (sb[-G:] == -7).all()
    t = tsb.cpu().numpy()
    assert (t[:4] == -3).all() and (t[5:] == -3).all()
    yb = ybuf.cpu().numpy()
    assert (yb[:G] == -5).all() and (yb[-G:] == -5).all()
    o = run_oracle(x_np, fmt, gran)
    assert np.array_equal(codes.cpu().numpy(), o["codes"])


def test_workspace_reuse_and_streams():
    """Back-to-back calls on one workspace and on a side stream give identical results."""
    import precision_quantization_gb300 as qz
    import torch
    x_np = gen(300, 512, "bf16", seed=800)
    x = to_device(x_np)
    ws = qz.Workspace()
    torch.cuda.synchronize()
    ref = None
    s = torch.cuda.Stream()
    for i in range(6):
        stream = s if i % 2 else None
        with torch.cuda.stream(s if stream else torch.cuda.current_stream()):
            q, st = qz.quantize(x, qz.QZ_NVFP4, "block", stats=True, workspace=ws, stream=stream)
        torch.cuda.synchronize()
        cur = (q.codes.cpu().numpy(), q.scales.cpu().numpy(), qz.read_stats(st))
        if ref is None:
            ref = cur
        assert np.array_equal(cur[0], ref[0]) and np.array_equal(cur[1], ref[1])
        assert cur[2] == ref[2]


# ------------------------------------------------------------------ the named workloads
CONFIG_RUNS = {
    1: [(O.INT8, O.GRAN_TENSOR), (O.E4M3, O.GRAN_TENSOR), (O.MXFP4, O.GRAN_BLOCK),
        (O.NVFP4, O.GRAN_BLOCK)],
    2: [(O.INT8, O.GRAN_ROW), (O.E4M3, O.GRAN_ROW), (O.MXFP4, O.GRAN_BLOCK),
        (O.NVFP4, O.GRAN_BLOCK)],
    3: [(O.E4M3, O.GRAN_ROW), (O.E5M2, O.GRAN_ROW), (O.NVFP4, O.GRAN_BLOCK)],
    4: [(O.MXFP4, O.GRAN_BLOCK), (O.NVFP4, O.GRAN_BLOCK)],
    5: [(f, g) for f in FMT8 for g in (O.GRAN_UNIT, O.GRAN_TENSOR)] +
       [(f, g) for f in FMT4 for g in (O.GRAN_UNIT, O.GRAN_BLOCK)],
}


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5])
def test_named_workload_full_size(k):
    """Every format of each named workload, at full size, against the oracle on the whole
    tensor (bf16 output for bf16 inputs, fp32 output for the fp32 edge mix)."""
    x = W.workload(k)
    od = ("f32",) if x.dtype == np.float32 else ("bf16",)
    for fmt, gran in CONFIG_RUNS[k]:
        g = run_gpu(x, fmt, gran, out_dtypes=od)
        o = run_oracle(x, fmt, gran, out_dtypes=od)
        assert_parity(g, o)
        assert g["status"] == 0
        if gran == O.GRAN_ROW:  # the quantize without statistics runs other kernels there
            assert_parity(run_gpu(x, fmt, gran, stats=False, out_dtypes=od), o, stats=False)


@pytest.mark.parametrize("fmt", FMT8)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_parity_row_with_stats_paths(fmt, dtype):
    """Per-row scales with the fused statistics: rows of a multiple of 4 whole chunks up to
    48 KiB take four warps each (a quarter row apiece); other rows of whole chunks up to
    16 KiB a warp and a shared-memory slot each; longer rows the row pipeline.  One-chunk
    rows, many short rows, rows of exactly 16 KiB and just past it, an odd row count, a
    single row of whole quarters, and rows of 32 and 48 KiB."""
    eb = 2 if dtype == "bf16" else 4
    shapes = [(1, 32 // eb), (3000, 64), (77, 4096 + 32), (9, 16384 // eb), (5, 16384 // eb + 32 // eb),
              (131, 1024), (1, 2048 // eb), (2, 32768 // eb), (7, 49152 // eb)]
    for i, (r, c) in enumerate(shapes):
        x = gen(r, c, dtype, seed=1100 + i, kind="edge" if (dtype == "f32" and i % 2) else "lognormal")
        assert_parity(run_gpu(x, fmt, O.GRAN_ROW), run_oracle(x, fmt, O.GRAN_ROW))


def test_row_with_stats_flags_nonfinite():
    """A NaN in one row of the warp-per-row path raises the non-finite flag."""
    x = W.lognormal_signed(40, 512, seed=1200, dtype="f32")
    x[17, 300] = np.float32("nan")
    g = run_gpu(x, O.E4M3, O.GRAN_ROW, out_dtypes=())
    assert g["status"] & 0x1
