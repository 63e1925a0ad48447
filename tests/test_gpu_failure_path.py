"""The staged kernels' failure path, exercised without a fault: a bounded wait that runs
out raises the status flag the host reads, and the context stays usable."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import assert_parity, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def test_pipeline_wait_limit_sets_status_and_context_survives():
    import time
    import precision_quantization_gb300 as qz
    import torch
    ws = qz.Workspace()
    assert ws.status() == 0
    t0 = time.perf_counter()
    assert qz.qz_selftest_pipeline_timeout(ws.ptr, 2_000_000) == qz.QZ_OK   # 2 ms limit
    flags = ws.status()
    elapsed = time.perf_counter() - t0
    assert flags & qz.QZ_FLAG_PIPELINE_TIMEOUT
    assert not flags & qz.QZ_FLAG_NONFINITE_INPUT
    assert elapsed < 5.0
    # the flag is sticky until the workspace is re-initialised
    assert ws.status() & qz.QZ_FLAG_PIPELINE_TIMEOUT
    ws.clear()
    assert ws.status() == 0
    # the context still runs the staged kernels correctly
    x = W.lognormal_signed(64, 4096, seed=801, sigma=2.0, dtype="f32")
    assert_parity(run_gpu(x, O.NVFP4, O.GRAN_BLOCK), run_oracle(x, O.NVFP4, O.GRAN_BLOCK))
    torch.cuda.synchronize()


def test_selftest_argument_errors():
    import precision_quantization_gb300 as qz
    ws = qz.Workspace()
    assert qz.qz_selftest_pipeline_timeout(None, 1000) == qz.QZ_ERR_WORKSPACE
    assert qz.qz_selftest_pipeline_timeout(ws.ptr, 0) == qz.QZ_ERR_UNSUPPORTED
    assert qz.qz_selftest_pipeline_timeout(ws.ptr, 10 ** 9) == qz.QZ_ERR_UNSUPPORTED
    assert qz.qz_selftest_pipeline_timeout(ws.ptr + 4, 1000) == qz.QZ_ERR_ALIGN
