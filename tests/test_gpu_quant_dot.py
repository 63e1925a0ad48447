"""GPU parity of the quantized matrix product (qz_quant_dot) against the oracle's exact
double sum: every output within E 2^-24 of the sum of the terms' magnitudes, with E the
bound include/qz.h derives from the operations of each form (gpu_util.qdot_bound); and
bit-exact equality where every partial sum is exact in fp32 (small integer activations,
power-of-two scales), which a dropped, doubled or misplaced term cannot pass."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import qdot_bound, qdot_tolerance, torch_mod

pytestmark = pytest.mark.gpu


def pack_words(vals):
    rows, n = vals.shape
    out = np.zeros((rows, (n + 7) // 8), dtype=np.uint32)
    for i in range(n):
        out[:, i // 8] |= vals[:, i].astype(np.uint32) << np.uint32(4 * (i % 8))
    return out


def make(n0, mid, group, n1, seed):
    rng = np.random.default_rng(seed)
    ng = mid // group
    w = pack_words(rng.integers(0, 16, (n0, mid)))
    sc = (rng.standard_normal((n0, ng)) * 0.02).astype(np.float32)
    sh = pack_words(rng.integers(0, 16, (n0, ng)))
    y = W.bf16_bits(W.normal(mid, max(n1, 1), 1.0, seed=seed + 1, dtype="f32"))[:, :n1]
    return w, sc, sh, np.ascontiguousarray(y)


@pytest.mark.parametrize("ypad,zpad", [(0, 0), (8, 3), (5, 0)])
@pytest.mark.parametrize("n0,mid,group,n1", [(1, 8, 8, 1), (7, 64, 16, 3), (33, 1024, 128, 8),
                                             (128, 4096, 32, 5), (5, 96, 12, 2), (64, 256, 256, 1),
                                             (300, 2048, 64, 4), (9, 520, 40, 7),
                                             (17, 96, 32, 8), (40, 192, 48, 6), (129, 8192, 128, 8),
                                             (260, 640, 16, 2)])
def test_quant_dot_parity(n0, mid, group, n1, ypad, zpad):
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    w, sc, sh, y = make(n0, mid, group, n1, seed=930 + n0 + mid)
    zr, za = O.quant_dot(w, sc, sh, y, group)
    yb = torch.zeros((mid, n1 + ypad), dtype=torch.int16, device="cuda")
    yb[:, :n1] = torch.from_numpy(y.view(np.int16)).cuda()
    yd = yb.view(torch.bfloat16)[:, :n1]
    zb = torch.full((n0, n1 + zpad), 7.0, dtype=torch.float32, device="cuda")
    z = qz.quant_dot(torch.from_numpy(w.view(np.int32)).cuda(), torch.from_numpy(sc).cuda(),
                     torch.from_numpy(sh.view(np.int32)).cuda(), group, yd, out=zb[:, :n1])
    torch.cuda.synchronize()
    got = z.cpu().numpy().astype(np.float64)
    tol = qdot_tolerance(mid, group, za)
    assert np.all(np.abs(got - zr) <= tol), float(np.max((np.abs(got - zr) - tol) / za))
    assert np.all(zb[:, n1:].cpu().numpy() == 7.0)  # nothing written past n1


def test_quant_dot_weight_like_shape():
    """A 4096 x 4096 weight (the weight-like workload's shape) in groups of 128, 8 columns."""
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    n0 = mid = 4096
    w, sc, sh, y = make(n0, mid, 128, 8, seed=950)
    zr, za = O.quant_dot(w, sc, sh, y, 128)
    z = qz.quant_dot(torch.from_numpy(w.view(np.int32)).cuda(), torch.from_numpy(sc).cuda(),
                     torch.from_numpy(sh.view(np.int32)).cuda(), 128,
                     torch.from_numpy(y.view(np.int16)).cuda().view(torch.bfloat16))
    got = z.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - zr) <= qdot_tolerance(mid, 128, za))


def make_exact(n0, mid, group, n1, seed):
    """Weights, power-of-two scales (1/4 .. 2), shifts and small-integer activations in
    [-4, 4]: every term is a multiple of 1/4 below 2^7 and every partial sum a multiple of
    1/4 below 2^20, all exact in fp32 whatever the order and the accumulator's rounding,
    so the GPU must give the oracle's sum bit for bit."""
    rng = np.random.default_rng(seed)
    ng = mid // group
    w = pack_words(rng.integers(0, 16, (n0, mid)))
    sc = (2.0 ** rng.integers(-2, 2, (n0, ng))).astype(np.float32)
    sh = pack_words(rng.integers(0, 16, (n0, ng)))
    yi = rng.integers(-4, 5, (mid, n1)).astype(np.float32)
    y = (yi.view(np.uint32) >> 16).astype(np.uint16)  # exact in bf16
    return w, sc, sh, np.ascontiguousarray(y)


@pytest.mark.parametrize("n0,mid,group,n1", [(129, 8192, 128, 8), (4096, 4096, 64, 8),
                                             (300, 2048, 16, 4), (33, 1024, 256, 8),
                                             (9, 520, 40, 7), (64, 96, 12, 1)])
def test_quant_dot_exact_sums(n0, mid, group, n1):
    """Tensor-core form (groups of 16 .. 256, split rows) and FMA form (groups of 40, 12):
    with every partial sum exact the result must equal the oracle's exactly."""
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    w, sc, sh, y = make_exact(n0, mid, group, n1, seed=970 + n0 + group)
    zr, _ = O.quant_dot(w, sc, sh, y, group)
    z = qz.quant_dot(torch.from_numpy(w.view(np.int32)).cuda(), torch.from_numpy(sc).cuda(),
                     torch.from_numpy(sh.view(np.int32)).cuda(), group,
                     torch.from_numpy(y.view(np.int16)).cuda().view(torch.bfloat16))
    got = z.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != zr)
    assert bad.size == 0, (len(bad), tuple(bad[0]), got[tuple(bad[0])], zr[tuple(bad[0])])


# ---- many activation columns: the tcgen05 tensor-memory product -------------------------
@pytest.mark.parametrize("ypad,zpad", [(0, 0), (8, 3), (5, 0)])
@pytest.mark.parametrize("n0,mid,group,n1", [(300, 1024, 128, 300), (128, 2048, 64, 256),
                                             (200, 4096, 16, 72), (64, 960, 48, 40),
                                             (130, 4096, 2048, 24), (257, 512, 256, 9),
                                             (40, 640, 32, 520)])
def test_quant_dot_many_columns_parity(n0, mid, group, n1, ypad, zpad):
    """Ragged tiles in both dimensions, groups that end inside a 64-wide step (16, 32, 48),
    groups longer than one accumulation piece (2048), split sums (few row tiles), padded
    rows of y and z, and an unaligned y row pitch (ypad 5: the column-block path)."""
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    w, sc, sh, y = make(n0, mid, group, n1, seed=990 + n0 + n1)
    zr, za = O.quant_dot(w, sc, sh, y, group)
    yb = torch.zeros((mid, n1 + ypad), dtype=torch.int16, device="cuda")
    yb[:, :n1] = torch.from_numpy(y.view(np.int16)).cuda()
    yd = yb.view(torch.bfloat16)[:, :n1]
    zb = torch.full((n0, n1 + zpad), 7.0, dtype=torch.float32, device="cuda")
    z = qz.quant_dot(torch.from_numpy(w.view(np.int32)).cuda(), torch.from_numpy(sc).cuda(),
                     torch.from_numpy(sh.view(np.int32)).cuda(), group, yd, out=zb[:, :n1])
    torch.cuda.synchronize()
    got = z.cpu().numpy().astype(np.float64)
    tol = qdot_tolerance(mid, group, za)
    assert np.all(np.abs(got - zr) <= tol), float(np.max((np.abs(got - zr) - tol) / za))
    assert np.all(zb[:, n1:].cpu().numpy() == 7.0)  # nothing written past n1


@pytest.mark.parametrize("n0,mid,group,n1", [(129, 8192, 128, 64), (300, 2048, 32, 300),
                                             (128, 1024, 1024, 256), (77, 4096, 2048, 33)])
def test_quant_dot_many_columns_exact_sums(n0, mid, group, n1):
    """Every partial sum exact in fp32: the tensor-memory product must equal the oracle bit
    for bit, whatever the accumulation order, so no term may be dropped, doubled or moved."""
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    w, sc, sh, y = make_exact(n0, mid, group, n1, seed=1010 + n0 + group)
    zr, _ = O.quant_dot(w, sc, sh, y, group)
    z = qz.quant_dot(torch.from_numpy(w.view(np.int32)).cuda(), torch.from_numpy(sc).cuda(),
                     torch.from_numpy(sh.view(np.int32)).cuda(), group,
                     torch.from_numpy(y.view(np.int16)).cuda().view(torch.bfloat16))
    got = z.cpu().numpy().astype(np.float64)
    bad = np.argwhere(got != zr)
    assert bad.size == 0, (len(bad), tuple(bad[0]), got[tuple(bad[0])], zr[tuple(bad[0])])


@pytest.mark.parametrize("n0,mid,group,n1", [(4096, 4096, 128, 4096), (32768, 8192, 128, 2048)])
def test_quant_dot_many_columns_full_size_sampled(n0, mid, group, n1):
    """The weight-like 4096 x 4096 weight with 4096 activation columns and the 32768 x 8192
    weight with 2048 columns (the bench's prefill cases), in the launch configuration the
    bench times: every output of 24 sampled rows x 40 sampled columns (the first and last
    rows and columns among them) against the oracle."""
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    rng = np.random.default_rng(1030 + n0)
    ng = mid // group
    codes = rng.integers(0, 2 ** 32, (n0, mid // 8), dtype=np.uint64).astype(np.uint32)
    sc = (rng.standard_normal((n0, ng)) * 0.02).astype(np.float32)
    sh = rng.integers(0, 2 ** 32, (n0, (ng + 7) // 8), dtype=np.uint64).astype(np.uint32)
    y = W.bf16_bits(W.normal(mid, n1, 1.0, seed=1031 + n0, dtype="f32"))
    z = qz.quant_dot(torch.from_numpy(codes.view(np.int32)).cuda(), torch.from_numpy(sc).cuda(),
                     torch.from_numpy(sh.view(np.int32)).cuda(), group,
                     torch.from_numpy(y.view(np.int16)).cuda().view(torch.bfloat16))
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([[0, n0 - 1], rng.integers(0, n0, 22)]))
    cols = np.unique(np.concatenate([[0, n1 - 1], rng.integers(0, n1, 38)]))
    zr, za = O.quant_dot(codes[rows], sc[rows], sh[rows], np.ascontiguousarray(y[:, cols]), group)
    got = z[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy()
    tol = qdot_tolerance(mid, group, za)
    assert np.all(np.abs(got.astype(np.float64) - zr) <= tol)


def test_quant_dot_many_columns_split_last_wave():
    """More tiles than SMs (154 tiles of 128 x 256 on a 152-SM GB300): the whole waves run as
    they are, and the tiles of the last, partly filled wave are split along l and added into
    z, which the library zeroes from the first split tile's row on.  Tile row 21 holds both
    whole tiles (stored) and split ones (added), and z starts as a sentinel.  Exact sums, so
    every sampled output must equal the oracle's bit for bit: the first rows, the last two
    tile rows whole, and every third column with the last."""
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    n0, mid, group, n1 = 22 * 128 - 50, 1024, 128, 7 * 256 - 10
    w, sc, sh, y = make_exact(n0, mid, group, n1, seed=1050)
    zb = torch.full((n0, n1), 7.0, dtype=torch.float32, device="cuda")
    z = qz.quant_dot(torch.from_numpy(w.view(np.int32)).cuda(), torch.from_numpy(sc).cuda(),
                     torch.from_numpy(sh.view(np.int32)).cuda(), group,
                     torch.from_numpy(y.view(np.int16)).cuda().view(torch.bfloat16), out=zb)
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(6), np.arange(20 * 128, n0)])
    cols = np.unique(np.concatenate([np.arange(0, n1, 3), [n1 - 1]]))
    zr, _ = O.quant_dot(w[rows], sc[rows], sh[rows], np.ascontiguousarray(y[:, cols]), group)
    got = z[torch.from_numpy(rows).cuda()][:, torch.from_numpy(cols).cuda()].cpu().numpy()
    bad = np.argwhere(got.astype(np.float64) != zr)
    assert bad.size == 0, (len(bad), tuple(bad[0]))
