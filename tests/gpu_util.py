"""Helpers for the GPU parity tests: run the CUDA path (through the C ABI binding) and the
CPU oracle on the same host array and compare them."""
from __future__ import annotations

import numpy as np

import oracle as O

BITEXACT_STATS_FIELDS = ("max_abs_err", "max_rel_err", "n")
STATS_RTOL = 1e-5  # sum of squares / MSE: compensated fp32 per thread, fp64 across threads


def torch_mod():
    import torch
    return torch


def to_device(x_np: np.ndarray, ld_pad: int = 0):
    """numpy (uint16 bf16 bits or float32) -> CUDA tensor, optionally as a view with a
    leading dimension of cols + ld_pad."""
    torch = torch_mod()
    rows, cols = x_np.shape
    if x_np.dtype == np.uint16:
        t = torch.from_numpy(np.ascontiguousarray(x_np).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x_np))
    t = t.cuda()
    if ld_pad:
        big = torch.zeros((rows, cols + ld_pad), dtype=t.dtype, device=t.device)
        big[:, :cols] = t
        t = big[:, :cols]
    return t


def to_host_bits(t) -> np.ndarray:
    torch = torch_mod()
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.contiguous().cpu().numpy().view(np.uint32)
    return t.contiguous().cpu().numpy()


def run_gpu(x_np, fmt, gran, scale_round=0, tensor_amax=None, stats=True, ld_pad=0,
            out_dtypes=("bf16", "f32"), block_size=None):
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    x = to_device(x_np, ld_pad)
    ws = qz.Workspace(x.device)
    ta = None
    if tensor_amax is not None:
        ta = torch.tensor([tensor_amax], dtype=torch.float32, device=x.device)
    q, st = qz.quantize(x, fmt, gran, scale_round, ta, stats=stats, workspace=ws,
                        block_size=block_size)
    ys = {}
    for od in out_dtypes:
        dt = torch.bfloat16 if od == "bf16" else torch.float32
        ys[od] = qz.dequantize(q, dt)
    st2 = qz.error_stats(x, q, ws) if stats else None
    torch.cuda.synchronize()
    out = dict(codes=to_host_bits(q.codes),
               scales=None if q.scales is None else to_host_bits(q.scales),
               ts=np.float32(q.tensor_scale.item()),
               y={k: to_host_bits(v) for k, v in ys.items()},
               status=ws.status())
    if stats:
        out["stats"] = qz.read_stats(st)
        out["stats2"] = qz.read_stats(st2)
    return out


def run_oracle(x_np, fmt, gran, scale_round=0, tensor_amax=None, stats=True,
               out_dtypes=("bf16", "f32"), block_size=None):
    rows, cols = x_np.shape
    codes, scales, ts, st = O.quantize(x_np, fmt, gran, scale_round, tensor_amax, stats,
                                       block_size=block_size)
    y = {}
    for od in out_dtypes:
        odt = O.BF16 if od == "bf16" else O.F32
        yy = O.dequantize(codes, scales, ts, fmt, gran, rows, cols, out_dtype=odt,
                          block_size=block_size)
        y[od] = yy if odt == O.BF16 else yy.view(np.uint32)
    if scales is not None and scales.dtype == np.float32:
        scales = scales.view(np.uint32)
    return dict(codes=codes, scales=scales, ts=ts, y=y, stats=st)


def _first_diff(a, b):
    idx = np.argwhere(a != b)
    return None if idx.size == 0 else (tuple(idx[0]), a[tuple(idx[0])], b[tuple(idx[0])], len(idx))


def assert_stats_close(s, o, what="stats"):
    for f in BITEXACT_STATS_FIELDS:
        assert getattr(s, f) == getattr(o, f), (what, f, getattr(s, f), getattr(o, f))
    for f in ("sum_sq_err", "mse"):
        a, b = getattr(s, f), getattr(o, f)
        if a == b:  # includes equal infinities (x^ past the binary32 range)
            continue
        assert abs(a - b) <= STATS_RTOL * abs(b) + 1e-300, (what, f, a, b)


def assert_parity(g, o, stats=True):
    d = _first_diff(g["codes"], o["codes"])
    assert d is None, f"codes differ at {d}"
    if o["scales"] is not None:
        d = _first_diff(g["scales"], o["scales"])
        assert d is None, f"scales differ at {d}"
    assert g["ts"].view(np.uint32) == o["ts"].view(np.uint32), (g["ts"], o["ts"])
    for k in o["y"]:
        d = _first_diff(g["y"][k], o["y"][k])
        assert d is None, f"dequantized ({k}) differs at {d}"
    if stats:
        assert_stats_close(g["stats"], o["stats"], "fused")
        assert_stats_close(g["stats2"], o["stats"], "standalone")


def qdot_bound(mid: int, group: int) -> int:
    """E of the quantized-product error bound in include/qz.h: every output is within
    E * 2^-24 * sum |terms| of the exact sum (tensor-core steps of 16 exact products with
    truncated alignment, plus one fp32 rounding per weight, group piece FMA, lane term and
    split partial)."""
    def cdiv(a, b):
        return -(-a // b)
    g = min(group, 1024)
    return 34 * cdiv(g, 16) + cdiv(mid, g) + cdiv(mid, 32) + cdiv(mid, 256) + 24


def qdot_tolerance(mid: int, group: int, zabs):
    """Absolute tolerance per output from the oracle's sum of term magnitudes (first-order
    bound times 1.001 for the second-order terms)."""
    return qdot_bound(mid, group) * 2.0 ** -24 * 1.001 * zabs + 1e-35
