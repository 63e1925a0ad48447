"""qz_error_stats_noalloc: the error statistics for callers that cannot allocate device
memory themselves (inside another framework's memory pool, on paths where cudaMalloc and
its device synchronisation are not allowed, or as a plugin handed only its buffers), so
cannot pass a workspace.  Its results must be those of qz_error_stats (which is given a
workspace) and of the oracle, on two calls in a row; qz_error_stats_noalloc_status must
report a non-finite input and start clean again after it has been read.

This file is collected last on purpose: a run that stops at the first failure has then
already run every other test.  The tests need no state from earlier tests and pass on
their own in a fresh process too."""
import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.gpu

# the oracle's own enumerators for the format and granularity names used here
OFMT = {"int8": O.INT8, "e4m3": O.E4M3, "e5m2": O.E5M2, "mxfp4": O.MXFP4, "nvfp4": O.NVFP4,
        "int4": O.INT4}
OGRAN = {"tensor": O.GRAN_TENSOR, "row": O.GRAN_ROW, "block": O.GRAN_BLOCK, "unit": O.GRAN_UNIT}

CASES = [("nvfp4", "block", "bf16", None, 0), ("mxfp4", "block", "f32", None, 0),
         ("int8", "row", "bf16", None, 0), ("e4m3", "tensor", "f32", None, 0),
         ("e5m2", "unit", "bf16", None, 0), ("int4", "block", "bf16", 32, 0),
         ("int4", "block", "f32", 128, 0), ("nvfp4", "block", "bf16", None, 24),
         ("mxfp4", "block", "bf16", None, 8), ("e4m3", "row", "f32", None, 3)]


def noalloc_stats(qz, x, q):
    """Call the entry point through the C ABI; returns the device qz_stats buffer."""
    import torch
    rows, cols, ld = qz._rows_cols_ld(x)
    desc = qz.make_desc(q.fmt, qz._dtype_code(x.dtype), q.granularity, rows, cols, ld,
                        block_size=q.block_size or None)
    stream = torch.cuda.current_stream().cuda_stream
    st = torch.full((qz.STATS_BYTES,), 0xAB, dtype=torch.uint8, device="cuda")
    rc = qz.qz_error_stats_noalloc(desc, x.data_ptr(), q.codes.data_ptr(), qz._ptr(q.scales),
                                   qz._ptr(q.tensor_scale), st.data_ptr(), stream)
    assert rc == qz.QZ_OK, qz.qz_status_string(rc)
    return st


@pytest.mark.parametrize("fmt,gran,dtype,bs,ld_pad", CASES)
def test_error_stats_noalloc_matches_workspace_path(fmt, gran, dtype, bs, ld_pad):
    import torch

    import precision_quantization_gb300 as qz
    import workloads as W
    from gpu_util import assert_stats_close, run_oracle, to_device

    x_np = W.lognormal_signed(300, 1024, seed=31, dtype=dtype)
    x = to_device(x_np, ld_pad)
    q, _ = qz.quantize(x, fmt, gran, block_size=bs)
    ref = qz.read_stats(qz.error_stats(x, q))  # existing entry point, caller-owned workspace
    orc = run_oracle(x_np, OFMT[fmt], OGRAN[gran], out_dtypes=(), block_size=bs)["stats"]
    stream = torch.cuda.current_stream().cuda_stream
    assert qz.qz_error_stats_noalloc_status(stream)[0] == qz.QZ_OK  # start from clean flags
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        st = noalloc_stats(qz, x, q)
        torch.cuda.synchronize()
        got = qz.read_stats(st)
        assert_stats_close(got, ref, "no-alloc vs workspace path")
        assert_stats_close(got, orc, "no-alloc vs oracle")
    assert qz.qz_error_stats_noalloc_status(stream) == (qz.QZ_OK, 0)


@pytest.mark.parametrize("fmt,gran", [("nvfp4", "block"), ("e4m3", "tensor"), ("int4", "block")])
def test_error_stats_noalloc_reports_nonfinite_input(fmt, gran):
    """A NaN in x raises QZ_FLAG_NONFINITE_INPUT, read (and cleared) by the status query;
    a clean call afterwards reports nothing, and its statistics are the oracle's."""
    import torch

    import precision_quantization_gb300 as qz
    import workloads as W
    from gpu_util import assert_stats_close, run_oracle, to_device

    x_np = W.lognormal_signed(64, 512, seed=33, dtype="f32")
    x = to_device(x_np)
    q, _ = qz.quantize(x, fmt, gran)
    stream = torch.cuda.current_stream().cuda_stream
    assert qz.qz_error_stats_noalloc_status(stream)[0] == qz.QZ_OK
    bad = x.clone()
    bad[5, 77] = float("nan")
    noalloc_stats(qz, bad, q)
    rc, flags = qz.qz_error_stats_noalloc_status(stream)
    assert rc == qz.QZ_OK and flags & qz.QZ_FLAG_NONFINITE_INPUT, flags
    st = noalloc_stats(qz, x, q)
    assert qz.qz_error_stats_noalloc_status(stream) == (qz.QZ_OK, 0)
    assert_stats_close(qz.read_stats(st), run_oracle(x_np, OFMT[fmt], OGRAN[gran], out_dtypes=())["stats"],
                       "no-alloc after a flagged call")


def test_error_stats_noalloc_argument_errors():
    import precision_quantization_gb300 as qz
    d = qz.make_desc("nvfp4", qz.QZ_BF16, "block", 4, 64)
    assert qz.lib().qz_error_stats_noalloc(None, 1, 1, 1, 1, 1, None) == qz.QZ_ERR_NULL
    assert qz.qz_error_stats_noalloc(d, 1 << 20, 1 << 20, 1 << 20, 1 << 20, None) == qz.QZ_ERR_NULL
    assert qz.lib().qz_error_stats_noalloc_status(None, None) == qz.QZ_ERR_NULL
