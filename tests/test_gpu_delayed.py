"""GPU parity of qz_quantize_delayed: the per-tensor scale comes from an amax handed in (a
previous tensor's), and the call returns this tensor's own amax.

Codes, scales and tensor scale must equal the oracle's quantization with that amax
supplied; the fused statistics must match it as in the other parity tests; the returned
amax must equal the oracle's max |x| bit for bit."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import assert_stats_close, to_device, to_host_bits, torch_mod

pytestmark = pytest.mark.gpu

RUNS = [(O.NVFP4, O.GRAN_BLOCK), (O.INT8, O.GRAN_TENSOR), (O.E4M3, O.GRAN_TENSOR),
        (O.E5M2, O.GRAN_TENSOR), (O.MXFP4, O.GRAN_BLOCK), (O.NVFP4, O.GRAN_UNIT),
        (O.INT8, O.GRAN_UNIT), (O.E4M3, O.GRAN_ROW)]


def needs_alpha(fmt, gran):
    return gran == O.GRAN_TENSOR or (fmt == O.NVFP4 and gran == O.GRAN_BLOCK)


def run_delayed(x_np, fmt, gran, amax_in, ld_pad=0, alias=False):
    """One call; returns the outputs and the amax it wrote.  alias: amax_in and amax_out
    are the same device word."""
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    x = to_device(x_np, ld_pad)
    ws = qz.Workspace(x.device)
    a_in = None
    if amax_in is not None:
        a_in = torch.tensor([amax_in], dtype=torch.float32, device=x.device)
    a_out = a_in if alias else None
    q, st, a_out = qz.quantize_delayed(x, fmt, a_in if needs_alpha(fmt, gran) or alias else None,
                                       gran, stats=True, workspace=ws, amax_out=a_out)
    torch.cuda.synchronize()
    return dict(codes=to_host_bits(q.codes),
                scales=None if q.scales is None else to_host_bits(q.scales),
                ts=np.float32(q.tensor_scale.item()), stats=qz.read_stats(st),
                amax=np.float32(a_out.item()), status=ws.status())


def check(g, x_np, fmt, gran, amax_in):
    codes, scales, ts, st = O.quantize(x_np, fmt, gran, O.SCALE_UP,
                                       amax_in if needs_alpha(fmt, gran) else None, True)
    assert np.array_equal(g["codes"], codes)
    if scales is not None:
        s = scales.view(np.uint32) if scales.dtype == np.float32 else scales
        assert np.array_equal(g["scales"], s)
    if needs_alpha(fmt, gran) or gran == O.GRAN_UNIT:
        assert g["ts"].view(np.uint32) == np.float32(ts).view(np.uint32)
    assert_stats_close(g["stats"], st, "fused")
    assert g["amax"].view(np.uint32) == np.float32(O.amax(x_np)).view(np.uint32)
    assert g["status"] == 0


@pytest.mark.parametrize("pad", [0, 24])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("fmt,gran", RUNS)
def test_delayed_parity(fmt, gran, dtype, pad):
    x = W.lognormal_signed(192, 1024, seed=620, sigma=2.0, dtype="f32")
    if dtype == "bf16":
        x = W.bf16_bits(x)
    a = float(np.float32(O.amax(x)))
    # the current tensor's own amax, a stale smaller one (saturation) and a larger one
    for factor in (1.0, 0.25, 3.0):
        amax_in = float(np.float32(a * factor))
        g = run_delayed(x, fmt, gran, amax_in, ld_pad=pad)
        check(g, x, fmt, gran, amax_in)


@pytest.mark.parametrize("fmt,gran", [(O.NVFP4, O.GRAN_BLOCK), (O.E4M3, O.GRAN_TENSOR)])
def test_delayed_chain_in_place(fmt, gran):
    """Step k uses step k-1's amax, with amax_in and amax_out in the same device word."""
    xs = [W.bf16_bits(W.lognormal_signed(64, 2048, seed=630 + k, sigma=2.0, dtype="f32") *
                      np.float32(4.0 ** k)) for k in range(3)]
    prev = float(np.float32(O.amax(xs[0]))) * 0.5
    for x in xs:
        g = run_delayed(x, fmt, gran, prev, alias=True)
        check(g, x, fmt, gran, prev)
        prev = float(g["amax"])


def test_delayed_full_size_stream():
    """The bench workload at full size: NVFP4 with the tensor's own amax supplied."""
    x = W.workload(4)
    a = float(np.float32(O.amax(x)))
    g = run_delayed(x, O.NVFP4, O.GRAN_BLOCK, a)
    check(g, x, O.NVFP4, O.GRAN_BLOCK, a)


def test_delayed_empty():
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    x = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    a_in = torch.tensor([5.0], dtype=torch.float32, device="cuda")
    q, st, a_out = qz.quantize_delayed(x, "nvfp4", a_in, "block", stats=True)
    torch.cuda.synchronize()
    assert a_out.item() == 0.0
    assert qz.read_stats(st).n == 0
