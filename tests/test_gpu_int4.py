"""GPU parity of grouped symmetric INT4 and of the asymmetric 4-bit group dequantization,
through the C ABI, against the CPU oracle: codes, group scales and dequantized values
bit-exact, max |e| and max |e|/|x| bit-exact, the sum of squares within 1e-5."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_util import assert_parity, run_gpu, run_oracle, to_host_bits, torch_mod

pytestmark = pytest.mark.gpu

GROUPS = [16, 32, 64, 128]


def gen(rows, cols, dtype, seed):
    x = W.lognormal_signed(rows, cols, seed=seed, sigma=2.0, dtype="f32")
    return W.bf16_bits(x) if dtype == "bf16" else x


@pytest.mark.parametrize("pad", [0, 24])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("bs", GROUPS)
def test_int4_parity(bs, dtype, pad):
    for rows, cols in [(1, bs), (3, 2 * bs), (33, 4 * bs), (257, 1024)]:
        x = gen(rows, cols, dtype, seed=700 + bs + rows)
        assert_parity(run_gpu(x, O.INT4, O.GRAN_BLOCK, ld_pad=pad, block_size=bs),
                      run_oracle(x, O.INT4, O.GRAN_BLOCK, block_size=bs))


@pytest.mark.parametrize("bs", [16, 128])
def test_int4_ties_zeros_and_extremes(bs):
    """Exact midpoints (k + 1/2) s, zero groups, signed zeros, denormals, and groups whose
    scale leaves the range of the FMA-corrected quotient."""
    rng = np.random.default_rng(710)
    x = np.zeros((8, 4 * bs), dtype=np.float32)
    s = np.float32(0.375)
    x[0, 0] = 7 * s                      # group scale exactly s
    x[0, 1:16] = (rng.integers(-7, 7, 15) + 0.5).astype(np.float32) * s   # ties
    x[1] = -0.0                          # a zero group (s := 1) with signed zeros
    x[2, :] = np.float32(-1e-42)
    x[3] = (rng.standard_normal(4 * bs) * 1e-39).astype(np.float32)
    x[4] = (rng.standard_normal(4 * bs) * 3e37).astype(np.float32)
    x[5] = (rng.standard_normal(4 * bs) * 1e-30).astype(np.float32)
    x[6] = rng.standard_normal(4 * bs).astype(np.float32)
    x[7, ::3] = np.float32(1e30)
    assert_parity(run_gpu(x, O.INT4, O.GRAN_BLOCK, block_size=bs),
                  run_oracle(x, O.INT4, O.GRAN_BLOCK, block_size=bs))


def test_int4_weight_like_full_size():
    """The weight-like workload (4096 x 4096 bf16, [out, in]) in groups of 128 along K."""
    x = W.workload(2)
    assert_parity(run_gpu(x, O.INT4, O.GRAN_BLOCK, block_size=128, out_dtypes=("bf16",)),
                  run_oracle(x, O.INT4, O.GRAN_BLOCK, block_size=128, out_dtypes=("bf16",)))


def pack_words(vals, per=8):
    """[rows, n] ints in 0..15 -> [rows, ceil(n/8)] uint32, element i in nibble i % 8."""
    rows, n = vals.shape
    nw = (n + per - 1) // per
    out = np.zeros((rows, nw), dtype=np.uint32)
    for i in range(n):
        out[:, i // per] |= vals[:, i].astype(np.uint32) << np.uint32(4 * (i % per))
    return out


@pytest.mark.parametrize("pad", [0, 8, 3])
@pytest.mark.parametrize("out", ["bf16", "f32"])
@pytest.mark.parametrize("rows,cols,group", [(1, 8, 8), (5, 64, 16), (7, 96, 12),
                                             (33, 1024, 128), (64, 4096, 32), (3, 40, 40)])
def test_asym4_parity(rows, cols, group, out, pad):
    import precision_quantization_gb300 as qz
    torch = torch_mod()
    rng = np.random.default_rng(720 + rows + group)
    codes = rng.integers(0, 16, (rows, cols))
    ng = cols // group
    w = pack_words(codes)
    sc = (rng.standard_normal((rows, ng)) * np.exp(rng.uniform(-8, 8, (rows, ng)))).astype(np.float32)
    sh = pack_words(rng.integers(0, 16, (rows, ng)))
    odt = O.BF16 if out == "bf16" else O.F32
    want = O.dequant_asym4(w, sc, sh, rows, cols, group, out_dtype=odt)
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    big = torch.zeros((rows, cols + pad), dtype=dt, device="cuda")
    y = big[:, :cols]
    wd = torch.from_numpy(w.view(np.int32)).cuda()
    shd = torch.from_numpy(sh.view(np.int32)).cuda()
    got = qz.dequantize_asym4(wd, torch.from_numpy(sc).cuda(), shd, group, out=y)
    torch.cuda.synchronize()
    g = to_host_bits(got)
    assert np.array_equal(g, want if out == "bf16" else want.view(np.uint32))
    assert not big[:, cols:].any()  # nothing written past the row
