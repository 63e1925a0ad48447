"""The calls can be recorded into a CUDA graph and replayed: they only enqueue kernels on
the caller's stream (no allocation, no synchronisation, launch parameters cached by an
earlier call), and the workspace's completion counters wrap back to zero after each
launch, so every replay starts from the same state."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import assert_stats_close, to_host_bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,gran", [(O.NVFP4, O.GRAN_BLOCK), (O.MXFP4, O.GRAN_BLOCK),
                                      (O.E4M3, O.GRAN_TENSOR), (O.INT4, O.GRAN_BLOCK)])
def test_graph_replay_matches_oracle(fmt, gran):
    import torch
    import precision_quantization_gb300 as qz
    rows, cols = 256, 4096
    xs = [W.bf16_bits(W.lognormal_signed(rows, cols, seed=900 + k, sigma=2.0, dtype="f32"))
          for k in range(3)]
    x = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    ws = qz.Workspace()
    codes, scales, ts = qz.alloc_outputs(fmt, gran, rows, cols, "cuda")
    st = torch.empty((qz.STATS_BYTES,), dtype=torch.uint8, device="cuda")
    y = torch.empty_like(x)
    d = qz.make_desc(fmt, qz.QZ_BF16, gran, rows, cols)

    def step(stream):
        sp = stream.cuda_stream
        assert qz.qz_quantize(d, x.data_ptr(), codes.data_ptr(), qz._ptr(scales), ts.data_ptr(),
                              None, st.data_ptr(), ws.ptr, sp) == 0
        assert qz.qz_dequantize(d, codes.data_ptr(), qz._ptr(scales), ts.data_ptr(), y.data_ptr(),
                                qz.QZ_BF16, sp) == 0

    x.copy_(torch.from_numpy(xs[0].view(np.int16)).view(torch.bfloat16))
    step(torch.cuda.current_stream())  # warm-up: launch parameters cached outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            step(side)
    for xn in xs:
        x.copy_(torch.from_numpy(xn.view(np.int16)).view(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        c, s, t, ost = O.quantize(xn, fmt, gran, stats=True)
        assert np.array_equal(to_host_bits(codes), c)
        if s is not None:
            sw = s.view(np.uint32) if s.dtype == np.float32 else s
            assert np.array_equal(to_host_bits(scales), sw)
        assert np.float32(ts.item()).view(np.uint32) == np.float32(t).view(np.uint32)
        yo = O.dequantize(c, s, t, fmt, gran, rows, cols, out_dtype=O.BF16)
        assert np.array_equal(to_host_bits(y), yo)
        assert_stats_close(qz.read_stats(st), ost, "graph replay")
    assert ws.status() == 0
