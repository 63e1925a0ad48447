"""Seeded synthetic inputs for the quantize / dequantize / error-statistics path.

This module only draws numbers: it holds none of the quantization arithmetic.  Both the
CPU oracle (in the tests and the CPU baseline) and the CUDA path are fed the very same
host arrays that these functions return.

Tensors are numpy arrays: bf16 tensors as ``np.uint16`` bit patterns (fp32 draws
converted to bf16 with round-to-nearest-even), fp32 tensors as ``np.float32``.

The five named workloads are the weight-like, activation-like and streaming tensors the
blog post "浅谈低精度浮点数" reasons about (weights with outliers tens of times the
typical magnitude, activations with outlier channels hundreds of times larger), plus an
fp32 edge-case mix for the element casts.  Large tensors are drawn in fixed row chunks,
each from its own child seed of ``numpy.random.SeedSequence(seed)``, so the result does
not depend on how many threads draw them.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

CHUNK_ELEMS = 1 << 22

WORKLOADS = {
    1: dict(name="iid-normal-1024x1024-bf16", rows=1024, cols=1024, dtype="bf16", seed=1),
    2: dict(name="weight-like-4096x4096-bf16", rows=4096, cols=4096, dtype="bf16", seed=2),
    3: dict(name="activation-like-8192x4096-bf16", rows=8192, cols=4096, dtype="bf16",
            seed=3),
    4: dict(name="lognormal-stream-32768x8192-bf16", rows=32768, cols=8192, dtype="bf16",
            seed=4),
    5: dict(name="edge-mix-16384x16384-f32", rows=16384, cols=16384, dtype="f32", seed=5),
}


# ------------------------------------------------------------------ helpers
def bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (inputs are finite)."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    out = np.empty(b.shape, dtype=np.uint16)
    step = CHUNK_ELEMS
    flat_b, flat_o = b.reshape(-1), out.reshape(-1)
    for i in range(0, flat_b.size, step):
        v = flat_b[i:i + step]
        flat_o[i:i + step] = ((v + (((v >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)
    return out


def _chunked(rows: int, cols: int, seed, fill, threads: int | None = None) -> np.ndarray:
    """Fill a float32 [rows, cols] array chunk by chunk; fill(rng, count) -> values."""
    out = np.empty((rows, cols), dtype=np.float32)
    if rows == 0 or cols == 0:
        return out
    rpc = max(1, CHUNK_ELEMS // cols)
    starts = list(range(0, rows, rpc))
    ss = seed if isinstance(seed, np.random.SeedSequence) else np.random.SeedSequence(seed)
    seeds = ss.spawn(len(starts))
    flat = out.reshape(-1)

    def work(i):
        r0 = starts[i]
        r1 = min(rows, r0 + rpc)
        rng = np.random.Generator(np.random.PCG64(seeds[i]))
        flat[r0 * cols:r1 * cols] = fill(rng, (r1 - r0) * cols)

    nthr = threads or min(16, os.cpu_count() or 1)
    if len(starts) == 1 or nthr == 1:
        for i in range(len(starts)):
            work(i)
    else:
        with cf.ThreadPoolExecutor(nthr) as ex:
            list(ex.map(work, range(len(starts))))
    return out


def _finish(a: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits(a) if dtype == "bf16" else a


# ------------------------------------------------------------------ distributions
def normal(rows: int, cols: int, std: float = 1.0, seed: int = 0, dtype: str = "bf16"):
    """i.i.d. N(0, std^2)."""
    def fill(rng, n):
        return (rng.standard_normal(n, dtype=np.float32) * np.float32(std)).astype(np.float32)
    return _finish(_chunked(rows, cols, seed, fill), dtype)


def weight_like(rows: int, cols: int, seed: int = 2, std: float = 0.02,
                frac: float = 0.001, factor: float = 50.0, dtype: str = "bf16"):
    """[out, in] weight: N(0, std^2) with a fraction of seeded positions scaled by factor."""
    base_ss, pos_ss = np.random.SeedSequence(seed).spawn(2)
    a = _chunked(rows, cols, base_ss,
                 lambda rng, n: rng.standard_normal(n, dtype=np.float32) * np.float32(std))
    n = rows * cols
    k = int(frac * n)
    if k:
        pos = np.random.Generator(np.random.PCG64(pos_ss)).choice(n, size=k, replace=False)
        a.reshape(-1)[pos] *= np.float32(factor)
    return _finish(a, dtype)


def activation_like(rows: int, cols: int, seed: int = 3, n_outlier: int = 8,
                    lo: float = 100.0, hi: float = 500.0, dtype: str = "bf16"):
    """[tokens, hidden] activations: N(0,1) with n_outlier seeded channels scaled by U[lo, hi]."""
    base_ss, col_ss = np.random.SeedSequence(seed).spawn(2)
    a = _chunked(rows, cols, base_ss,
                 lambda rng, n: rng.standard_normal(n, dtype=np.float32))
    rng = np.random.Generator(np.random.PCG64(col_ss))
    k = min(n_outlier, cols)
    chans = rng.choice(cols, size=k, replace=False)
    factors = rng.uniform(lo, hi, size=k).astype(np.float32)
    a[:, chans] *= factors[None, :]
    return _finish(a, dtype)


def lognormal_signed(rows: int, cols: int, seed: int = 4, sigma: float = 2.0,
                     dtype: str = "bf16"):
    """|x| = exp(N(0, sigma^2)), sign +-1 with probability 1/2 each."""
    def fill(rng, n):
        z = rng.standard_normal(n, dtype=np.float32)
        sgn = rng.integers(0, 2, n, dtype=np.int8)
        v = np.exp(np.float32(sigma) * z)
        return np.where(sgn == 1, -v, v).astype(np.float32)
    return _finish(_chunked(rows, cols, seed, fill), dtype)


# Finite non-negative value sets of the element grids, from the format definitions
# (INT8 integers 0..127; E4M3 bias 7 without Inf, max 448; E5M2 bias 15, max 57344;
# E2M1 bias 1).  Used only to place exact round-to-nearest ties in the edge-case mix.
def _grid_values(fmt: str) -> np.ndarray:
    if fmt == "int8":
        return np.arange(128, dtype=np.float64)
    if fmt == "e2m1":
        return np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], dtype=np.float64)
    mbits, bias, emax = {"e4m3": (3, 7, 15), "e5m2": (2, 15, 30)}[fmt]
    vals = [m / 2 ** mbits * 2.0 ** (1 - bias) for m in range(2 ** mbits)]
    for e in range(1, emax + 1):
        for m in range(2 ** mbits):
            if fmt == "e4m3" and e == 15 and m == 7:
                continue
            vals.append((1 + m / 2 ** mbits) * 2.0 ** (e - bias))
    return np.array(sorted(vals), dtype=np.float64)


_GRIDS = ("int8", "e4m3", "e5m2", "e2m1")
_MAXES = np.array([127.0, 448.0, 57344.0, 6.0])
_SUBNORMAL_TOP = np.array([2.0 ** -6, 2.0 ** -14, 1.0])  # E4M3, E5M2, E2M1 subnormal ranges


def _midpoints() -> np.ndarray:
    mids = []
    for g in _GRIDS:
        v = _grid_values(g)
        mids.append(((v[:-1] + v[1:]) / 2).astype(np.float32))
    return mids


def edge_mix(rows: int, cols: int, seed: int = 5):
    """fp32 edge-case mix, per element (category drawn i.i.d., which shuffles positions):
    50% N(0,1); 20% exact midpoints between neighbouring grid values of INT8 / E4M3 /
    E5M2 / E2M1 (a quarter each, both signs); 10% the FP8 / E2M1 subnormal ranges and
    fp32 denormals; 10% beyond a format maximum (1-100x INT8 / E4M3 / E5M2 / E2M1 max, one
    in five log-uniform in [1e30, 3e38]); 10% zeros, half of them -0."""
    mids = _midpoints()

    def fill(rng, n):
        u = rng.random(n)
        out = rng.standard_normal(n, dtype=np.float32)
        sign = np.where(rng.random(n) < 0.5, np.float32(-1), np.float32(1))
        # exact ties
        t = (u >= 0.5) & (u < 0.7)
        nt = int(t.sum())
        which = rng.integers(0, 4, nt)
        vals = np.empty(nt, dtype=np.float32)
        for g in range(4):
            sel = which == g
            vals[sel] = mids[g][rng.integers(0, mids[g].size, int(sel.sum()))]
        out[t] = vals * sign[t]
        # subnormal ranges
        s = (u >= 0.7) & (u < 0.8)
        ns = int(s.sum())
        kind = rng.integers(0, 4, ns)
        sv = np.empty(ns, dtype=np.float32)
        for g in range(3):
            sel = kind == g
            sv[sel] = (rng.random(int(sel.sum())) * _SUBNORMAL_TOP[g]).astype(np.float32)
        sel = kind == 3
        mant = rng.integers(1, 1 << 23, int(sel.sum()), dtype=np.uint32)
        sv[sel] = mant.view(np.float32)  # exponent field 0: fp32 denormals
        out[s] = sv * sign[s]
        # beyond the format maximum
        b = (u >= 0.8) & (u < 0.9)
        nb = int(b.sum())
        f = 10.0 ** rng.uniform(0.0, 2.0, nb)
        bv = (f * _MAXES[rng.integers(0, 4, nb)])
        huge = rng.random(nb) < 0.2
        bv[huge] = 10.0 ** rng.uniform(30.0, np.log10(3e38), int(huge.sum()))
        out[b] = bv.astype(np.float32) * sign[b]
        # zeros, half negative
        z = u >= 0.9
        out[z] = np.where(rng.random(int(z.sum())) < 0.5, np.float32(-0.0), np.float32(0.0))
        return out

    return _chunked(rows, cols, seed, fill)


def workload(k: int, rows: int | None = None, cols: int | None = None) -> np.ndarray:
    """Input of named workload k (1..5); rows/cols override the shape (same recipe)."""
    w = WORKLOADS[k]
    r = w["rows"] if rows is None else rows
    c = w["cols"] if cols is None else cols
    s = w["seed"]
    if k == 1:
        return normal(r, c, 1.0, s)
    if k == 2:
        return weight_like(r, c, s)
    if k == 3:
        return activation_like(r, c, s)
    if k == 4:
        return lognormal_signed(r, c, s)
    if k == 5:
        return edge_mix(r, c, s)
    raise KeyError(k)
