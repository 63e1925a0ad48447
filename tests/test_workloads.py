"""Seeded input generators: determinism and the stated structure of each workload."""
import numpy as np

import workloads as W


def test_deterministic_and_thread_independent():
    a = W.lognormal_signed(300, 8192, seed=4)
    b = W.lognormal_signed(300, 8192, seed=4)
    assert np.array_equal(a, b)
    c = W._chunked(300, 8192, 4, lambda rng, n: rng.standard_normal(n, dtype=np.float32),
                   threads=1)
    d = W._chunked(300, 8192, 4, lambda rng, n: rng.standard_normal(n, dtype=np.float32),
                   threads=8)
    assert np.array_equal(c, d)


def test_bf16_bits_rne():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3e38], dtype=np.float32)
    h = W.bf16_bits(x)
    back = (h.astype(np.uint32) << 16).view(np.float32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: goes to the even one (1.0)
    assert list(back[:4]) == [1.0, 1.0, 1.015625, -2.5]


def test_weight_like_outliers():
    x = W.weight_like(256, 256, seed=2)
    f = (x.astype(np.uint32) << 16).view(np.float32)
    k = int(0.001 * 256 * 256)
    assert np.sum(np.abs(f) > 0.02 * 6) >= k * 0.9   # the scaled positions stand out


def test_activation_like_outlier_channels():
    x = W.activation_like(512, 128, seed=3)
    f = (x.astype(np.uint32) << 16).view(np.float32)
    colmax = np.abs(f).max(axis=0)
    assert np.sum(colmax > 50) == 8


def test_edge_mix_categories():
    x = W.edge_mix(64, 4096, seed=5)
    n = x.size
    zeros = np.sum(x == 0)
    neg_zero = np.sum((x == 0) & np.signbit(x))
    assert 0.08 * n < zeros < 0.12 * n and 0.3 * zeros < neg_zero < 0.7 * zeros
    denorm = np.sum((x != 0) & (np.abs(x) < np.float32(1.1754944e-38)))
    assert denorm > 0.01 * n
    assert np.sum(np.abs(x) > 1e30) > 0.001 * n
    # exact midpoints of the E2M1 grid appear
    assert np.sum(np.isin(np.abs(x), np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]))) > 0
    assert np.all(np.isfinite(x))


def test_named_shapes():
    for k, w in W.WORKLOADS.items():
        x = W.workload(k, rows=8, cols=w["cols"])
        assert x.shape == (8, w["cols"])
        assert x.dtype == (np.uint16 if w["dtype"] == "bf16" else np.float32)
