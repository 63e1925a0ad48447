"""The CPU oracle pinned to what the blog post "浅谈低精度浮点数" fixes.

Each test checks the oracle against a value the post prints (tests/golden/*.json, each
with its citation), a closed form, an invariant, or brute force on small inputs --
never against a re-typed copy of the oracle's own formula.
"""
import math

import numpy as np
import pytest

from conftest import golden

def f32(v):
    return np.float32(v)


# ---------------------------------------------------------------- binary32 / bf16
def test_ieee754_worked_example(orc):
    g = golden("ieee754_worked_example.json")
    bits = int(g["all_bits"], 2)
    assert bits == int(g["hex"], 16)
    assert orc.decode_fp32(bits) == g["value"]
    assert orc.encode_fp32(g["value"]) == bits
    # field split of the printed bit string
    assert bits >> 31 == g["sign"]
    assert (bits >> 23) & 0xFF == g["biased_exponent"] == int(g["biased_exponent_bits"], 2)
    assert bits & 0x7FFFFF == int(g["fraction_bits"], 2)
    assert g["biased_exponent"] - g["bias"] == 4  # 1.1001001 x 2^4


def test_fp32_range(orc):
    g = golden("fp32_range.json")
    mx = orc.decode_fp32(0x7F7FFFFF)
    mn = orc.decode_fp32(0x00800000)
    assert f"{mx:.7e}" == "3.4028235e+38"
    assert f"{mn:.8e}" == "1.17549435e-38"
    assert mx == (2 - 2 ** -23) * 2.0 ** g["normal_exponent_max"]
    assert mn == 2.0 ** g["normal_exponent_min"]
    sub = orc.decode_fp32(0x00000001)
    assert 0 < sub < mn  # subnormals exist below the smallest normal
    assert math.isinf(orc.decode_fp32(0x7F800000))
    assert math.isnan(orc.decode_fp32(0x7FC00000))
    assert orc.decode_fp32(0x80000000) == 0 and math.copysign(1, orc.decode_fp32(0x80000000)) < 0


def test_fp32_encode_decode_roundtrip_random(orc):
    rng = np.random.default_rng(11)
    for b in rng.integers(0, 1 << 32, 3000, dtype=np.uint64):
        b = int(b)
        if (b >> 23) & 0xFF == 0xFF:
            continue
        assert orc.encode_fp32(orc.decode_fp32(b)) == b


def test_bf16_layout_is_fp32_top_half(orc):
    """BF16 has fp32's 8 exponent bits and 7 fraction bits: the two independently
    written decoders must agree on every finite bf16 code."""
    g = golden("fp32_range.json")
    assert g["bf16_exponent_bits"] + g["bf16_fraction_bits"] + 1 == 16
    for h in range(0, 1 << 16, 7):
        if (h >> 7) & 0xFF == 0xFF:
            continue
        assert orc.decode_bf16(h) == orc.decode_fp32(h << 16)


def test_bf16_rne_brute_force(orc):
    """fp32 -> bf16 picks the nearer of the two neighbouring bf16 values, ties to the one
    with an even last fraction bit (checked with exact double arithmetic)."""
    rng = np.random.default_rng(12)
    cases = [int(b) for b in rng.integers(0, 0x7F7F0000, 4000, dtype=np.uint64)]
    cases += [0x3F808000, 0x3F818000, 0x00008000, 0x00018000, 0x7F7F7FFF, 0x00000001]
    for b in cases:
        v = orc.decode_fp32(b)
        lo_bits = b & 0xFFFF0000
        lo, hi = orc.decode_fp32(lo_bits), orc.decode_fp32(lo_bits + 0x10000)
        h = orc.bf16_rne(b)
        got = orc.decode_bf16(h)
        dl, dh = v - lo, hi - v
        if dl < dh:
            want = lo
        elif dh < dl:
            want = hi
        else:
            want = lo if ((lo_bits >> 16) & 1) == 0 else hi
        assert got == want, hex(b)
        # sign symmetry
        assert orc.bf16_rne(b | 0x80000000) == (h | 0x8000)


# ---------------------------------------------------------------- element formats
def _finite_codes(orc, fmt, n):
    out = []
    for c in range(n):
        v = orc.decode_code(fmt, c)
        if math.isfinite(v):
            out.append((c, v))
    return out


def test_e2m1_value_set(orc):
    g = golden("e2m1_values.json")
    vals = sorted(orc.decode_code(orc.E2M1, c) for c in range(16))
    want = sorted(g["values"] + [-0.0])
    assert vals == want
    assert orc.decode_code(orc.E2M1, 0x8) == 0 and math.copysign(1, orc.decode_code(orc.E2M1, 8)) < 0


def test_e4m3_max_and_nan(orc):
    g = golden("fp8_facts.json")
    fin = _finite_codes(orc, orc.E4M3, 256)
    assert max(v for _, v in fin) == g["e4m3_max"] == 448.0
    assert orc.decode_code(orc.E4M3, 0x7E) == 448.0          # S.1111.110 = 1.75 * 2^8
    assert math.isnan(orc.decode_code(orc.E4M3, 0x7F))       # S.1111.111 is NaN, no Inf
    assert math.isnan(orc.decode_code(orc.E4M3, 0xFF))
    assert len(fin) == 254


def test_e5m2_ieee_like(orc):
    """Reading (the post gives no E5M2 specials): IEEE-like, max 57344, field 31 = Inf/NaN."""
    fin = _finite_codes(orc, orc.E5M2, 256)
    assert max(v for _, v in fin) == 57344.0
    assert math.isinf(orc.decode_code(orc.E5M2, 0x7C))
    assert all(math.isnan(orc.decode_code(orc.E5M2, c)) for c in (0x7D, 0x7E, 0x7F))
    assert len(fin) == 248


@pytest.mark.parametrize("fmt,lo,hi,key", [
    ("E4M3", 2, 4, "e4m3_values_in_2_4"),
    ("E5M2", 2, 4, "e5m2_values_in_2_4"),
    ("E5M2", 4, 8, "e5m2_values_in_4_8"),
])
def test_samples_per_binade(orc, fmt, lo, hi, key):
    g = golden("fp8_facts.json")
    f = getattr(orc, fmt)
    vals = {v for _, v in _finite_codes(orc, f, 128)}
    assert len([v for v in vals if lo <= v < hi]) == g[key]


def test_e8m0_powers_of_two(orc):
    for c in range(255):
        assert orc.decode_code(orc.E8M0, c) == 2.0 ** (c - 127)
    assert math.isnan(orc.decode_code(orc.E8M0, 255))


@pytest.mark.parametrize("fmt,n", [("E4M3", 256), ("E5M2", 256), ("E2M1", 16)])
def test_roundtrip_every_finite_code(orc, fmt, n):
    f = getattr(orc, fmt)
    for c, v in _finite_codes(orc, f, n):
        assert orc.encode_elem(f, v) == c, (fmt, hex(c), v)


def test_roundtrip_int8(orc):
    for q in range(-127, 128):
        assert orc.encode_elem(orc.INT8, float(q)) == (q & 0xFF)
    # -128 is never produced: the symmetric range is [-127, 127]
    g = golden("int8_facts.json")
    assert orc.decode_code(orc.INT8, orc.encode_elem(orc.INT8, -128.0)) == g["qmin"]
    assert orc.decode_code(orc.INT8, orc.encode_elem(orc.INT8, 1e6)) == g["qmax"]


def _brute_nearest(table_codes, table_vals, a):
    d = np.abs(np.asarray(table_vals) - a)
    best = np.flatnonzero(d == d.min())
    if len(best) == 1:
        return table_codes[best[0]]
    ev = [table_codes[i] for i in best if table_codes[i] % 2 == 0]
    assert len(ev) == 1
    return ev[0]


@pytest.mark.parametrize("fmt,n,signbit", [("E4M3", 127, 0x80), ("E5M2", 124, 0x80),
                                           ("E2M1", 8, 0x8), ("INT8", 128, None)])
def test_rne_saturating_brute_force(orc, fmt, n, signbit):
    """Nearest value by exhaustive search over the table, ties to an even code,
    saturation at the maximum, sign kept (INT8: two's complement)."""
    f = getattr(orc, fmt)
    codes = list(range(n))
    vals = [orc.decode_code(f, c) for c in codes]
    vmax = max(vals)
    rng = np.random.default_rng(13)
    xs = list(rng.uniform(0, vmax * 1.3, 1500).astype(np.float32))
    mids = [np.float32((vals[i] + vals[i + 1]) / 2) for i in range(n - 1)]
    xs += mids + [np.float32(v) for v in vals] + [np.float32(vmax * 2), np.float32(3e38)]
    for x in xs:
        a = float(x)
        want = codes[-1] if a >= vmax else _brute_nearest(codes, vals, a)
        assert orc.encode_elem(f, x) == want, (fmt, a)
        neg = orc.encode_elem(f, -x)
        if signbit is None:
            assert neg == ((-want) & 0xFF)
        else:
            assert neg == (want | signbit)


def test_ties_to_even_examples(orc):
    assert [orc.decode_code(orc.INT8, orc.encode_elem(orc.INT8, v))
            for v in (0.5, 1.5, 2.5, -0.5, -2.5, 126.5)] == [0, 2, 2, 0, -2, 126]
    e2m1 = [orc.decode_code(orc.E2M1, orc.encode_elem(orc.E2M1, v))
            for v in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)]
    assert e2m1 == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0]


def test_signed_zero(orc):
    assert orc.encode_elem(orc.E4M3, -0.0) == 0x80
    assert orc.encode_elem(orc.E5M2, -1e-30) == 0x80
    assert orc.encode_elem(orc.E2M1, -0.1) == 0x8
    assert orc.encode_elem(orc.INT8, -0.3) == 0x00


def test_rounding_is_monotone(orc):
    rng = np.random.default_rng(14)
    xs = np.sort(rng.uniform(-500, 500, 4000).astype(np.float32))
    for f in (orc.E4M3, orc.E5M2, orc.E2M1, orc.INT8):
        dec = [orc.decode_code(f, orc.encode_elem(f, x)) for x in xs]
        assert all(a <= b for a, b in zip(dec, dec[1:]))


# ---------------------------------------------------------------- error bounds (section FP8)
@pytest.mark.parametrize("fmt,mbits,key,lo_exp,hi_val", [
    ("E4M3", 3, "e4m3_rel_error_bound", -6, 448.0),
    ("E5M2", 2, "e5m2_rel_error_bound", -14, 57344.0),
])
def test_fp8_relative_error_bound(orc, fmt, mbits, key, lo_exp, hi_val):
    """|x - x^|/|x| <= 2^-(M+1) over the normal range, brute force over every fp32 value
    of one binade plus random fp32 values across the whole normal range."""
    g = golden("fp8_facts.json")
    bound = g[key]
    assert bound == 2.0 ** -(mbits + 1) == 2.0 ** -(g[fmt.lower() + "_mantissa_bits"] + 1)
    f = getattr(orc, fmt)
    # every fp32 in [1, 2) with a stride, and random values over [2^lo_exp, max]
    xs = [orc.decode_fp32(0x3F800000 + m) for m in range(0, 1 << 23, 97)]
    rng = np.random.default_rng(15)
    xs += list(np.exp2(rng.uniform(lo_exp, math.log2(hi_val), 4000)).astype(np.float32))
    worst = 0.0
    for x in xs:
        q = orc.decode_code(f, orc.encode_elem(f, x))
        worst = max(worst, abs(float(x) - q) / float(x))
    assert worst <= bound
    assert worst > 0.9 * bound / (1 + bound)  # the bound is attained up to the 1/(1+2^-(M+1)) factor


def test_int8_abs_error_bound(orc):
    """|x - x^| <= s/2 = alpha/254 (up to the binary32 rounding of s and x/s)."""
    g = golden("int8_facts.json")
    rng = np.random.default_rng(16)
    x = rng.standard_normal((64, 256)).astype(np.float32)
    codes, _, s, st = orc.quantize(x, orc.INT8, orc.GRAN_TENSOR, stats=True)
    alpha = float(np.abs(x).max())
    assert s == np.float32(np.float32(alpha) / np.float32(g["scale_divisor"]))
    q = codes.view(np.int8).astype(np.float64)
    assert q.min() >= g["qmin"] and q.max() <= g["qmax"]
    err = np.abs(x.astype(np.float64) - q * float(s))
    assert err.max() <= alpha / g["abs_error_divisor"] * (1 + 2 ** -20)
    assert float(st.max_abs_err) <= alpha / g["abs_error_divisor"] * (1 + 2 ** -20)


def test_int8_vs_e4m3_crossover(orc):
    """The INT8 relative error is bounded by alpha/(254|x|), which meets E4M3's 1/16 at
    |x| = 16 alpha/254 ~ 0.063 alpha.  Measured on the oracle (alpha = 1 through a
    per-tensor scale): the error never exceeds the bound, reaches it at the rounding
    midpoints, and the largest |x| whose INT8 error exceeds 1/16 lies just below
    0.063 alpha; over the same range E4M3 stays within 1/16."""
    g = golden("int8_facts.json")
    u_star = g["crossover_fraction_of_alpha"]
    assert abs(u_star - 16 / 254) < 5e-4
    bound = g["e4m3_rel_bound_used_for_crossover"]
    xs = np.linspace(0.01, 0.3, 200001).astype(np.float32)
    x = np.concatenate([xs, [np.float32(1.0)]])[None, :]
    codes, _, s, _ = orc.quantize(x, orc.INT8, orc.GRAN_TENSOR)
    q = codes.view(np.int8)[0, :-1].astype(np.float64)
    xf = xs.astype(np.float64)
    rel = np.abs(xf - q * float(s)) / xf
    env = 1.0 / (g["abs_error_divisor"] * xf)          # alpha / (254 |x|), alpha = 1
    assert np.all(rel <= env * (1 + 1e-5))
    k = np.arange(1, 30)
    mids = ((k + 0.5) * float(s)).astype(np.float32)
    xm = np.concatenate([mids, [np.float32(1.0)]])[None, :]
    cm, _, _, _ = orc.quantize(xm, orc.INT8, orc.GRAN_TENSOR)
    rm = np.abs(mids - cm.view(np.int8)[0, :-1] * float(s)) / mids
    assert np.allclose(rm, 1.0 / (2 * k + 1), rtol=1e-5)   # bound attained at midpoints
    last = xf[rel > bound].max()
    assert 0.9 * u_star <= last <= u_star
    assert np.all(rel[xf > u_star] < bound)
    ce, _, se, _ = orc.quantize(x, orc.E4M3, orc.GRAN_TENSOR)
    dq = np.array([orc.decode_code(orc.E4M3, int(c)) for c in ce[0, :-1:97]]) * float(se)
    assert np.max(np.abs(xf[::97] - dq) / xf[::97]) <= bound


def test_int8_zero_amax(orc):
    x = np.zeros((3, 40), dtype=np.float32)
    x[1, 3] = -0.0
    codes, _, s, st = orc.quantize(x, orc.INT8, orc.GRAN_TENSOR, stats=True)
    assert s == 1.0 and not codes.any()
    assert st.sum_sq_err == 0 and st.max_rel_err == 0


def test_saturation(orc):
    assert orc.encode_elem(orc.E4M3, 1000.0) == 0x7E
    assert orc.encode_elem(orc.E4M3, 464.0) == 0x7E     # would round past 448: saturates
    assert orc.encode_elem(orc.E5M2, 1e6) == 0x7B
    assert orc.encode_elem(orc.E5M2, 61440.0) == 0x7B   # IEEE would give Inf here
    assert orc.encode_elem(orc.E2M1, 100.0) == 0x7
    assert orc.encode_elem(orc.E2M1, -7.0) == 0xF
    assert orc.encode_elem(orc.INT8, 300.0) == 127


# ---------------------------------------------------------------- MXFP4
def test_mxfp4_worked_example(orc):
    g = golden("mxfp4_facts.json")
    for ex in g["example"]:
        t = np.float32(ex["a_over_6"])
        k = orc.mx_scale_exponent(t)
        assert 2.0 ** k == ex["scale"]
        # through the full quantizer: a block whose amax is A = 6 * (A/6)
        A = np.float32(t * np.float32(6))
        assert abs(float(A) / 6 - ex["a_over_6"]) < 1e-6
        x = np.zeros((1, 32), dtype=np.float32)
        x[0, 5] = A
        _, sc, _, _ = orc.quantize(x, orc.MXFP4, orc.GRAN_BLOCK)
        assert orc.decode_code(orc.E8M0, int(sc[0, 0])) == ex["scale"]


def test_mxfp4_scale_brute_force(orc):
    """UP: 2^(k-1) < t <= 2^k.  NEAREST: |log2 t - k| <= 1/2."""
    rng = np.random.default_rng(17)
    ts = np.exp2(rng.uniform(-120, 120, 3000)).astype(np.float32)
    ts = np.concatenate([ts, np.exp2(np.arange(-120, 121)).astype(np.float32)])
    for t in ts:
        k = orc.mx_scale_exponent(t, orc.SCALE_UP)
        assert 2.0 ** (k - 1) < float(t) <= 2.0 ** k
        kn = orc.mx_scale_exponent(t, orc.SCALE_NEAREST)
        assert abs(math.log2(float(t)) - kn) <= 0.5
    assert orc.mx_scale_exponent(np.float32(0)) == -127
    assert orc.mx_scale_exponent(np.float32(2.0 ** -140)) == -127  # clamped to E8M0 range


def _blocks(orc, fmt, x, **kw):
    codes, sc, ts, _ = orc.quantize(x, fmt, orc.GRAN_BLOCK, **kw)
    rows, cols = x.shape
    bs = orc.block_of(fmt)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(rows, cols)
    q = np.vectorize(lambda c: orc.decode_code(orc.E2M1, int(c)))(nib)
    if fmt == orc.MXFP4:
        s = np.vectorize(lambda c: orc.decode_code(orc.E8M0, int(c)))(sc)
    else:
        s = np.vectorize(lambda c: orc.decode_code(orc.E4M3, int(c)))(sc) * float(ts)
    s_el = np.repeat(s, bs, axis=1)
    A = np.abs(x.astype(np.float64)).reshape(rows, cols // bs, bs).max(-1)
    return q, s, s_el, A


def test_mxfp4_rho_error_and_zero_threshold(orc):
    g = golden("mxfp4_facts.json")
    rng = np.random.default_rng(18)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-20, 20, (64, 1)))).astype(np.float32)
    q, s, s_el, A = _blocks(orc, orc.MXFP4, x)
    rho = s / (A / 6)
    assert rho.min() >= g["rho_min"] and rho.max() < g["rho_max_exclusive"]
    e = np.abs(x - q * s_el)
    assert np.all(e <= s_el)                                   # |e| <= s
    Ael = np.repeat(A, 32, axis=1)
    assert np.all(e < Ael / 3)                                 # < A/3 in every case
    aligned = np.repeat(rho == 1.0, 32, axis=1)
    assert np.all(e[aligned] <= Ael[aligned] / 6)
    # zero threshold 0.25 s, between A/24 and A/12
    zt = g["zero_threshold_factor_of_scale"] * s
    frac = zt / A
    assert frac.min() >= g["zero_threshold_min_fraction_of_A"] - 1e-4
    assert frac.max() <= g["zero_threshold_max_fraction_of_A"] + 1e-4
    zt_el = np.repeat(zt, 32, axis=1)
    assert np.all(q[np.abs(x) < zt_el] == 0)
    assert np.all(np.abs(q[np.abs(x) > zt_el]) > 0)


def test_mxfp4_zero_threshold_tie(orc):
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0] = 6.0      # A = 6 -> t = 1 -> s = 1
    x[0, 1] = 0.25     # exactly 0.25 s: tie between 0 and 0.5 -> 0 (even code)
    x[0, 2] = np.nextafter(np.float32(0.25), np.float32(1))
    q, s, _, _ = _blocks(orc, orc.MXFP4, x)
    assert s[0, 0] == 1.0 and q[0, 1] == 0 and q[0, 2] == 0.5


# ---------------------------------------------------------------- NVFP4
def test_nvfp4_scales(orc):
    g = golden("nvfp4_facts.json")
    rng = np.random.default_rng(19)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.uniform(-3, 3, (64, 1)))).astype(np.float32)
    codes, sc, ts, _ = orc.quantize(x, orc.NVFP4, orc.GRAN_BLOCK)
    amax = float(np.abs(x).max())
    assert ts == np.float32(np.float32(amax) / np.float32(g["global_divisor"]))
    assert g["global_divisor"] == g["e2m1_max"] * g["e4m3_max"]
    # the block that holds the global amax gets the largest E4M3 block scale, 448
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert orc.decode_code(orc.E4M3, int(sc[r, c // 16])) == 448.0
    q, s, s_el, A = _blocks(orc, orc.NVFP4, x)
    rho = s / (A / 6)
    # block scales in the E4M3 normal range (>= 2^-6) have neighbour ratio <= 9/8
    normal = np.vectorize(lambda c: orc.decode_code(orc.E4M3, int(c)))(sc) >= 2.0 ** -6
    assert rho[normal].min() >= 1.0 and rho[normal].max() <= g["rho_max"] * (1 + 1e-6)
    e = np.abs(x - q * s_el)
    Ael = np.repeat(A, 16, axis=1)
    nel = np.repeat(normal, 16, axis=1)
    assert np.all(e[nel] <= g["abs_error_fraction_of_A"] * Ael[nel] * (1 + 1e-6))
    zt = 0.25 * s
    assert np.all((zt / A)[normal] <= g["zero_threshold_max_fraction_of_A"])


def test_nvfp4_block_scale_brute_force(orc):
    vals = [(c, orc.decode_code(orc.E4M3, c)) for c in range(127)]
    rng = np.random.default_rng(20)
    ts = list(np.exp2(rng.uniform(-12, 10, 3000)).astype(np.float32)) + \
        [np.float32(v) for _, v in vals] + [np.float32(500), np.float32(0)]
    for t in ts:
        up = orc.nv_block_scale_code(t, orc.SCALE_UP)
        if float(t) >= 448:
            assert up == 0x7E
        else:
            want = min((v, c) for c, v in vals if v >= float(t))[1]
            assert up == want
        ne = orc.nv_block_scale_code(t, orc.SCALE_NEAREST)
        assert ne == orc.encode_elem(orc.E4M3, t)


def test_nvfp4_unit_and_zero_blocks(orc):
    x = np.zeros((2, 32), dtype=np.float32)
    x[0, :16] = -0.0
    x[1, :] = np.linspace(-7, 7, 32, dtype=np.float32)
    codes, sc, ts, _ = orc.quantize(x, orc.NVFP4, orc.GRAN_BLOCK)
    assert sc[0, 0] == 0 and np.all(codes[0, :8] == 0x88)    # zero block: signed zeros
    codes_u, sc_u, ts_u, _ = orc.quantize(x, orc.NVFP4, orc.GRAN_UNIT)
    assert ts_u == 1.0 and np.all(sc_u == 0x38)
    assert orc.decode_code(orc.E2M1, int(codes_u[1, 0] & 0xF)) == -6.0   # -7 saturates


# ---------------------------------------------------------------- packing and stats
def test_nibble_order(orc):
    g = golden("nibble_order.json")
    assert g["first_element"] == "low nibble"
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, 0], x[0, 1], x[0, 2], x[0, 3] = 0.5, 1.0, -6.0, 3.0
    codes, _, _, _ = orc.quantize(x, orc.MXFP4, orc.GRAN_UNIT)
    assert codes[0, 0] == (0x2 << 4) | 0x1     # element 0 -> bits [0,4), element 1 -> [4,8)
    assert codes[0, 1] == (0x5 << 4) | 0xF


def test_stats_closed_form(orc):
    """x = [1, 1.0625] to E4M3 with unit scale: 1.0625 is the midpoint of 1 and 1.125,
    ties to 1 (even mantissa), so e = [0, 0.0625]."""
    x = np.array([[1.0, 1.0625]], dtype=np.float32)
    codes, _, _, st = orc.quantize(x, orc.E4M3, orc.GRAN_UNIT, stats=True)
    assert list(codes[0]) == [0x38, 0x38]
    assert st.sum_sq_err == 0.0625 ** 2 and st.mse == 0.0625 ** 2 / 2
    assert st.max_abs_err == np.float32(0.0625)
    assert st.max_rel_err == np.float32(np.float32(0.0625) / np.float32(1.0625))
    assert st.n == 2


def test_fused_and_standalone_stats_agree(orc):
    rng = np.random.default_rng(21)
    x = rng.standard_normal((17, 64)).astype(np.float32)
    for fmt, gran in [(orc.INT8, orc.GRAN_ROW), (orc.E5M2, orc.GRAN_TENSOR),
                      (orc.MXFP4, orc.GRAN_BLOCK), (orc.NVFP4, orc.GRAN_BLOCK)]:
        codes, sc, ts, st = orc.quantize(x, fmt, gran, stats=True)
        st2 = orc.error_stats(x, codes, sc, ts, fmt, gran)
        assert st == st2


def test_dequantize_matches_decode_times_scale(orc):
    rng = np.random.default_rng(22)
    x = rng.standard_normal((5, 48)).astype(np.float32)
    codes, sc, ts, _ = orc.quantize(x, orc.NVFP4, orc.GRAN_BLOCK)
    y = orc.dequantize(codes, sc, ts, orc.NVFP4, orc.GRAN_BLOCK, 5, 48, out_dtype=orc.F32)
    q, s, s_el, _ = _blocks(orc, orc.NVFP4, x)
    want = (q.astype(np.float32) * s_el.astype(np.float32)).astype(np.float32)
    assert np.array_equal(y.view(np.uint32), want.view(np.uint32))
    yb = orc.dequantize(codes, sc, ts, orc.NVFP4, orc.GRAN_BLOCK, 5, 48, out_dtype=orc.BF16)
    assert np.array_equal(yb, np.vectorize(lambda b: orc.bf16_rne(int(b)))(want.view(np.uint32)))


def test_unit_roundtrip_idempotent(orc):
    rng = np.random.default_rng(23)
    x = (rng.standard_normal((8, 64)) * 30).astype(np.float32)
    for fmt in (orc.INT8, orc.E4M3, orc.E5M2, orc.MXFP4, orc.NVFP4):
        codes, sc, ts, _ = orc.quantize(x, fmt, orc.GRAN_UNIT)
        y = orc.dequantize(codes, sc, ts, fmt, orc.GRAN_UNIT, 8, 64, out_dtype=orc.F32)
        codes2, _, _, _ = orc.quantize(y, fmt, orc.GRAN_UNIT)
        assert np.array_equal(codes, codes2)


def test_row_scale_and_ld(orc):
    rng = np.random.default_rng(24)
    base = rng.standard_normal((6, 40)).astype(np.float32)
    view = base[:, :33]          # ld 40 > cols 33
    codes, sc, _, st = orc.quantize(view, orc.E4M3, orc.GRAN_ROW, stats=True)
    for r in range(6):
        assert sc[r] == np.float32(np.abs(view[r]).max() / np.float32(448))
    dense = np.ascontiguousarray(view)
    codes2, sc2, _, st2 = orc.quantize(dense, orc.E4M3, orc.GRAN_ROW, stats=True)
    assert np.array_equal(codes, codes2) and np.array_equal(sc, sc2) and st == st2


def test_nonfinite_rejected(orc):
    x = np.ones((2, 32), dtype=np.float32)
    x[1, 7] = np.inf
    with pytest.raises(orc.OracleError):
        orc.quantize(x, orc.E4M3, orc.GRAN_TENSOR)


def test_empty(orc):
    x = np.zeros((0, 32), dtype=np.float32)
    codes, sc, ts, st = orc.quantize(x, orc.NVFP4, orc.GRAN_BLOCK, stats=True)
    assert codes.size == 0 and st.n == 0 and st.mse == 0 and ts == 1.0


# ---------------------------------------------------------------- INT4 (symmetric, grouped)
def test_int4_code_table(orc):
    """4-bit two's complement nibbles; symmetric quantization never produces -8."""
    g = golden("int4_facts.json")
    vals = [orc.decode_code(orc.INT4, c) for c in range(16)]
    assert vals == [float(v) for v in list(range(0, 8)) + list(range(-8, 0))]
    for q in range(g["qmin"], g["qmax"] + 1):
        assert orc.encode_elem(orc.INT4, float(q)) == (q & 0xF)
    assert orc.encode_elem(orc.INT4, -100.0) == (g["qmin"] & 0xF)   # saturates at -7, not -8
    assert orc.encode_elem(orc.INT4, 100.0) == g["qmax"]


def test_int4_rounding_brute_force(orc):
    """Element codes are round-half-to-even of v, clamped to [-7, 7] (numpy's rint)."""
    rng = np.random.default_rng(41)
    v = np.concatenate([rng.uniform(-9, 9, 4000), np.arange(-9, 9.5, 0.5)]).astype(np.float32)
    for x in v:
        q = int(np.clip(np.rint(np.float64(x)), -7, 7))
        assert orc.encode_elem(orc.INT4, float(x)) == (q & 0xF), x


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_int4_scale_bound_and_zero_threshold(orc, bs):
    """s = A/7 per group: the group's largest element maps to +-7, |e| <= s/2 = A/14, and
    |x| below the zero threshold A/14 (= s/2; the tie itself goes to the even 0) gives 0."""
    g = golden("int4_facts.json")
    assert abs(g["zero_threshold_fraction_of_A"] - 1 / g["abs_error_divisor"]) < 5e-5
    rng = np.random.default_rng(40 + bs)
    x = (rng.standard_normal((8, 4 * bs)) * np.exp(rng.uniform(-3, 3, (8, 1)))).astype(np.float32)
    codes, scales, _, st = orc.quantize(x, orc.INT4, orc.GRAN_BLOCK, stats=True, block_size=bs)
    assert scales.shape == (8, 4) and scales.dtype == np.float32
    q = (codes[:, :, None] >> np.array([0, 4], dtype=np.uint8)) & 0xF
    q = q.reshape(8, 4 * bs).astype(np.int64)
    q = np.where(q >= 8, q - 16, q)
    assert q.min() >= g["qmin"] and q.max() <= g["qmax"]
    xg = x.reshape(8, 4, bs).astype(np.float64)
    A = np.abs(xg).max(axis=2)
    assert np.array_equal(scales, (A.astype(np.float32) / np.float32(g["scale_divisor"])))
    qg = q.reshape(8, 4, bs)
    top = np.abs(xg).argmax(axis=2)
    assert np.all(np.abs(np.take_along_axis(qg, top[..., None], 2)) == g["qmax"])
    err = np.abs(xg - qg * scales[..., None].astype(np.float64))
    assert np.all(err <= A[..., None] / g["abs_error_divisor"] * (1 + 2 ** -20))
    s = scales[..., None].astype(np.float64)
    zero = np.abs(xg) < s / 2
    assert np.all(qg[zero] == 0)
    assert np.all(qg[np.abs(xg) > s / 2 * (1 + 2 ** -20)] != 0)
    # the tie x = s/2 rounds to the even integer 0; 3s/2 to 2
    xt = np.zeros((1, bs), dtype=np.float32)
    xt[0, 0], xt[0, 1], xt[0, 2] = 7.0, 0.5, 1.5
    ct, st_, _, _ = orc.quantize(xt, orc.INT4, orc.GRAN_BLOCK, block_size=bs)
    assert st_[0, 0] == 1.0 and ct[0, 0] == 0x07 and ct[0, 1] == 0x02


def test_int4_zero_group_and_dequantize(orc):
    x = np.zeros((2, 64), dtype=np.float32)
    x[1, 32:] = np.linspace(-3, 3, 32, dtype=np.float32)
    codes, scales, ts, st = orc.quantize(x, orc.INT4, orc.GRAN_BLOCK, stats=True)
    assert scales[0, 0] == 1.0 and not codes[0].any()              # A = 0: s := 1, codes 0
    y = orc.dequantize(codes, scales, ts, orc.INT4, orc.GRAN_BLOCK, 2, 64, out_dtype=orc.F32)
    nib = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(2, 64).astype(np.int64)
    nib = np.where(nib >= 8, nib - 16, nib)
    s = np.repeat(scales, 32, axis=1)
    assert np.array_equal(y, (nib.astype(np.float32) * s).astype(np.float32))
    st2 = orc.error_stats(x, codes, scales, ts, orc.INT4, orc.GRAN_BLOCK)
    assert st2 == st


# ---------------------------------------------------------------- Puzzle 12: asymmetric 4-bit
def test_asym4_worked_example(orc):
    g = golden("puzzle12_asym_dequant.json")
    ex = g["example"]
    w = np.array([ex["w_words"]], dtype=np.uint32)
    y = orc.dequant_asym4(w, np.array([[ex["scale"]]], dtype=np.float32),
                          np.array([[ex["shift"]]], dtype=np.uint32), 1, 16, ex["group"])
    assert y[0].tolist() == ex["y"]


def test_asym4_identity_order_and_groups(orc):
    """sc = 1, sh = 0 returns the packed codes themselves, in the puzzle's nibble order; each
    element uses the scale and shift of group c // group (shifts packed 8 per word)."""
    g = golden("nibble_order.json")
    assert g["first_element"] == "low nibble"
    rng = np.random.default_rng(44)
    rows, cols, group = 3, 256, 16
    codes = rng.integers(0, 16, (rows, cols))
    w = np.zeros((rows, cols // 8), dtype=np.uint32)
    for j in range(8):
        w |= (codes[:, j::8].astype(np.uint32) << np.uint32(4 * j))
    ng = cols // group
    y = orc.dequant_asym4(w, np.ones((rows, ng), np.float32), np.zeros((rows, 2), np.uint32),
                          rows, cols, group)
    assert np.array_equal(y, codes.astype(np.float32))
    # per-group powers of two and shifts: exact, so every element is checkable by hand
    sc = (2.0 ** rng.integers(-4, 5, (rows, ng))).astype(np.float32)
    shv = rng.integers(0, 16, (rows, ng))
    sh = np.zeros((rows, 2), dtype=np.uint32)
    for j in range(ng):
        sh[:, j // 8] |= shv[:, j].astype(np.uint32) << np.uint32(4 * (j % 8))
    y = orc.dequant_asym4(w, sc, sh, rows, cols, group)
    gi = np.arange(cols) // group
    assert np.array_equal(y, (sc[:, gi] * (codes - shv[:, gi])).astype(np.float32))
    yb = orc.dequant_asym4(w, sc, sh, rows, cols, group, out_dtype=orc.BF16)
    assert np.array_equal(yb, (y.view(np.uint32) >> 16).astype(np.uint16))  # exact in bf16


def test_quant_dot_worked_example(orc):
    g = golden("puzzle12_asym_dequant.json")
    ex, dx = g["example"], g["dot_example"]
    w = np.array([ex["w_words"]], dtype=np.uint32)
    y = np.full((16, 1), 0x3F80, dtype=np.uint16)          # bf16 1.0
    z, za = orc.quant_dot(w, np.array([[ex["scale"]]], np.float32),
                          np.array([[ex["shift"]]], np.uint32), y, ex["group"])
    assert z[0, 0] == dx["z"]
    assert za[0, 0] == sum(abs(v) for v in ex["y"])


def test_quant_dot_integer_and_dyadic_exact(orc):
    """With small integers (sc = 1, sh = 0) the product is an integer matrix product; with
    power-of-two scales and shifts every term and sum is a small dyadic rational, exact in
    float64, so numpy's matmul of the dequantized matrix gives the exact answer."""
    rng = np.random.default_rng(45)
    n0, mid, n1, group = 6, 128, 5, 32
    codes = rng.integers(0, 16, (n0, mid))
    w = np.zeros((n0, mid // 8), dtype=np.uint32)
    for j in range(8):
        w |= codes[:, j::8].astype(np.uint32) << np.uint32(4 * j)
    yi = rng.integers(-8, 9, (mid, n1))
    y = (np.float32(1.0) * yi).astype(np.float32).view(np.uint32) >> 16   # exact in bf16
    y = y.astype(np.uint16)
    ng = mid // group
    z, za = orc.quant_dot(w, np.ones((n0, ng), np.float32), np.zeros((n0, 1), np.uint32), y, group)
    assert np.array_equal(z, (codes @ yi).astype(np.float64))
    assert np.array_equal(za, (np.abs(codes) @ np.abs(yi)).astype(np.float64))
    sc = (2.0 ** rng.integers(-3, 4, (n0, ng))).astype(np.float32)
    shv = rng.integers(0, 16, (n0, ng))
    sh = np.zeros((n0, 1), dtype=np.uint32)
    for j in range(ng):
        sh[:, 0] |= shv[:, j].astype(np.uint32) << np.uint32(4 * j)
    gi = np.arange(mid) // group
    deq = sc[:, gi].astype(np.float64) * (codes - shv[:, gi])
    z, _ = orc.quant_dot(w, sc, sh, y, group)
    assert np.array_equal(z, deq @ yi.astype(np.float64))


def test_quant_dot_bound_catches_one_dropped_term(orc):
    """The tolerance the GPU parity tests allow (include/qz.h's E 2^-24 sum|terms|) is
    smaller than one term of average size at the full-size shapes, so a kernel that drops
    or doubles a single term fails.  Checked by planting the mistake in the oracle's
    inputs: zero one weight code's term by setting its code to its group's shift."""
    from gpu_util import qdot_tolerance
    rng = np.random.default_rng(46)
    for n0, mid, group, n1 in ((4, 8192, 128, 8), (4, 4096, 128, 8), (4, 4096, 64, 2)):
        ng = mid // group
        codes = rng.integers(0, 16, (n0, mid))
        shv = rng.integers(0, 16, (n0, ng))
        sc = (rng.standard_normal((n0, ng)) * 0.02).astype(np.float32)

        def pack(v):
            out = np.zeros((v.shape[0], (v.shape[1] + 7) // 8), dtype=np.uint32)
            for i in range(v.shape[1]):
                out[:, i // 8] |= v[:, i].astype(np.uint32) << np.uint32(4 * (i % 8))
            return out
        yf = rng.standard_normal((mid, n1)).astype(np.float32)
        y = (yf.view(np.uint32) >> 16).astype(np.uint16)
        z, za = orc.quant_dot(pack(codes), sc, pack(shv), y, group)
        tol = qdot_tolerance(mid, group, za)
        # drop, in every row, the term whose magnitude is the row's median (a typical term)
        c2 = codes.copy()
        for j in range(n0):
            gi = np.arange(mid) // group
            mag = np.abs(sc[j, gi] * (codes[j] - shv[j, gi]) * yf[:, 0].astype(np.float64))
            l = int(np.argsort(mag)[mid // 2])
            c2[j, l] = shv[j, l // group]
        z2, _ = orc.quant_dot(pack(c2), sc, pack(shv), y, group)
        assert np.all(np.abs(z2[:, 0] - z[:, 0]) > tol[:, 0]), (n0, mid, group)
