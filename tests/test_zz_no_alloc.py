"""qz_error_stats_noalloc: the error statistics for callers that cannot allocate device
memory themselves, so cannot pass a workspace.  Its results must be those of
qz_error_stats (which is given a workspace), on two calls in a row.

This file is collected last on purpose: a run that stops at the first failure has then
already run every other test.  The test needs no state from earlier tests and passes on
its own in a fresh process too."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,gran,dtype", [("nvfp4", "block", "bf16"), ("mxfp4", "block", "f32"),
                                            ("int8", "row", "bf16"), ("e4m3", "tensor", "f32"),
                                            ("e5m2", "unit", "bf16")])
def test_error_stats_noalloc_matches_workspace_path(fmt, gran, dtype):
    import torch

    import precision_quantization_gb300 as qz
    import workloads as W
    from gpu_util import assert_stats_close, to_device

    x_np = W.lognormal_signed(300, 1024, seed=31, dtype=dtype)
    x = to_device(x_np)
    q, _ = qz.quantize(x, fmt, gran)
    ref = qz.read_stats(qz.error_stats(x, q))  # existing entry point, caller-owned workspace
    rows, cols, ld = qz._rows_cols_ld(x)
    desc = qz.make_desc(q.fmt, qz._dtype_code(x.dtype), q.granularity, rows, cols, ld)
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # the second call reuses the scratch the first one left behind
        st = torch.full((qz.STATS_BYTES,), 0xAB, dtype=torch.uint8, device="cuda")
        rc = qz.qz_error_stats_noalloc(desc, x.data_ptr(), q.codes.data_ptr(), qz._ptr(q.scales),
                                       qz._ptr(q.tensor_scale), st.data_ptr(), stream)
        assert rc == qz.QZ_OK, qz.qz_status_string(rc)
        torch.cuda.synchronize()
        assert_stats_close(qz.read_stats(st), ref, "no-alloc")


def test_error_stats_noalloc_argument_errors():
    import precision_quantization_gb300 as qz
    d = qz.make_desc("nvfp4", qz.QZ_BF16, "block", 4, 64)
    assert qz.lib().qz_error_stats_noalloc(None, 1, 1, 1, 1, 1, None) == qz.QZ_ERR_NULL
    assert qz.qz_error_stats_noalloc(d, 1 << 20, 1 << 20, 1 << 20, 1 << 20, None) == qz.QZ_ERR_NULL
