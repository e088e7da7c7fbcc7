"""Pins of the oracle's exp / reciprocal / SiLU definition (its fused
multiply-add against exact rational arithmetic, accuracy against long-double
exp and float64 SiLU, limits fixed by the mathematics) and of the chained
SwiGLU requantization (hand-worked blocks, gate/up order, grouping)."""
import math
from fractions import Fraction

import numpy as np

from oracle import formats as F
from oracle import layout as L
from oracle import quantize as Q
from oracle import swiglu as S
from tests._golden import cases


def _round_f32_exact(q):
    """Nearest-even fp32 value of the exact rational q (as a Python float),
    written from the definition: the quantum 2^(e - 23) of q's binade
    (subnormal binade below 2^-126), round half to even, overflow to inf."""
    if q == 0:
        return 0.0
    sign = -1.0 if q < 0 else 1.0
    q = abs(q)
    e = q.numerator.bit_length() - q.denominator.bit_length()
    if Fraction(2) ** e > q:
        e -= 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    m = q / quantum
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = fl * quantum
    if v >= Fraction(2) ** 128:
        return sign * math.inf
    return sign * float(v)


def test_fma_f32_double_rounding_case():
    """a * b + c = 0.75 + 2^-25 + 2^-61: just above the midpoint between
    0.75 and 0.75 + 2^-24.  Rounding the float64 sum to nearest first lands
    on the midpoint (and then on 0.75); one rounding gives 0.75 + 2^-24."""
    a = np.float32((1 + 2.0 ** -12) * 2.0 ** -25)
    b = np.float32(1 - 2.0 ** -12 + 2.0 ** -24)
    c = np.float32(0.75)
    assert float(a) * float(b) == 2.0 ** -25 + 2.0 ** -61
    assert np.float32(np.float64(a) * np.float64(b) + np.float64(c)) == 0.75
    assert S.fma_f32(a, b, c) == np.float32(0.75 + 2.0 ** -24)


def test_fma_f32_against_exact_rationals():
    rng = np.random.default_rng(41)
    n = 3000
    a = (rng.standard_normal(n) * 2.0 ** rng.integers(-30, 30, n)).astype(np.float32)
    b = (rng.standard_normal(n) * 2.0 ** rng.integers(-30, 30, n)).astype(np.float32)
    c = (rng.standard_normal(n) * 2.0 ** rng.integers(-60, 60, n)).astype(np.float32)
    # cancellation: c close to -a*b
    k = n // 3
    c[:k] = -(a[:k].astype(np.float64) * b[:k]).astype(np.float32)
    c[k:2 * k] = np.nextafter(c[:k], np.float32(np.inf))
    # subnormal and tiny results
    a[-50:] = np.float32(2.0 ** -75)
    b[-50:] = rng.uniform(0.5, 1.0, 50).astype(np.float32) * np.float32(2.0 ** -60)
    c[-50:] = np.float32(0.0)
    got = S.fma_f32(a, b, c)
    for i in range(n):
        exact = Fraction(float(a[i])) * Fraction(float(b[i])) + Fraction(float(c[i]))
        assert float(got[i]) == _round_f32_exact(exact), (i, a[i], b[i], c[i])


def test_exp_neg_spec_accuracy_vs_long_double():
    x = np.concatenate([np.linspace(-87.0, 0.0, 400001),
                        -F.decode_bf16(np.arange(0x0000, 0x42AE, 3))]).astype(np.float32)
    got = S.exp_neg_spec(x).astype(np.longdouble)
    ref = np.exp(x.astype(np.longdouble))
    rel = np.abs(got - ref) / ref
    assert rel.max() <= 2.0 ** -22, float(rel.max())


def test_exp_neg_spec_special_points():
    assert S.exp_neg_spec(np.float32(0.0)) == 1.0
    assert S.exp_neg_spec(np.float32(-0.0)) == 1.0
    assert S.exp_neg_spec(np.float32(-104.0)) == 0.0
    assert S.exp_neg_spec(np.float32(-1e30)) == 0.0
    assert S.exp_neg_spec(np.float32(-np.inf)) == 0.0
    assert S.exp_neg_spec(np.float32(np.nan)) == 0.0
    # 2^n below 2^-126 is taken as 0: x log2(e) = -126.52 rounds to n = -127
    assert S.exp_neg_spec(np.float32(-87.7)) == 0.0
    # n = -126: a normal result close to e^x
    v = float(S.exp_neg_spec(np.float32(-87.3)))
    assert v >= 2.0 ** -126 and abs(v - math.exp(float(np.float32(-87.3)))) / v < 2.0 ** -22


def test_recip_spec_accuracy():
    d = np.arange(0x3F800000, 0x40000001, 3, dtype=np.uint32).view(np.float32)
    d = np.concatenate([d, np.float32([1.0, 1.5, 2.0])])
    r = S.recip_spec(d).astype(np.float64)
    ref = 1.0 / d.astype(np.float64)
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(r - ref) / ulp) <= 0.51
    assert S.recip_spec(np.float32(1.0)) == 1.0
    assert S.recip_spec(np.float32(2.0)) == 0.5


def test_silu_limits():
    z = S.silu_spec(np.float32(0.0))
    assert z == 0.0 and not np.signbit(z)
    z = S.silu_spec(np.float32(-0.0))
    assert z == 0.0 and np.signbit(z)
    assert S.silu_spec(np.float32(32.0)) == 32.0
    assert S.silu_spec(np.float32(1000.0)) == 1000.0
    assert S.silu_spec(np.float32(np.inf)) == np.inf
    assert np.isnan(S.silu_spec(np.float32(np.nan)))
    r = S.silu_spec(np.float32(-200.0))
    assert r == 0.0 and np.signbit(r)
    g = np.linspace(-60, 60, 20001).astype(np.float32)
    ref = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64)))
    got = S.silu_spec(g).astype(np.float64)
    big = np.abs(ref) > 1e-30
    assert np.max(np.abs(got[big] - ref[big]) / np.abs(ref[big])) < 2.0 ** -21


def test_silu_every_bf16_input():
    """Every finite bf16 gate value (the fused and chained paths feed SiLU
    bf16 numbers): within 2^-21 relative of float64 SiLU wherever that is
    above 1e-30, and -0 / 0 below (e^-|g| under 2^-126 is flushed)."""
    g = F.decode_bf16(np.arange(0, 65536)).astype(np.float32)
    g = g[np.isfinite(g)]
    got = S.silu_spec(g).astype(np.float64)
    with np.errstate(over="ignore"):
        ref = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64)))
    big = np.abs(ref) > 1e-30
    assert np.max(np.abs(got[big] - ref[big]) / np.abs(ref[big])) < 2.0 ** -21
    assert np.all(np.abs(got[~big]) <= 1e-30)


def test_silu_bf16_tails_reduce_exactly():
    """The kernels tabulate silu for bf16 gates with biased exponents 102..133
    and use two closed forms outside that band; every bf16 value (NaN and inf
    included) must give the definition's bits: g * 1/2 below exponent 102
    (|g| < 2^-25: e^-|g| rounds to 1, sigma to 1/2) and g * (1 if g >= 0 else
    0) above exponent 133 (|g| >= 128: e^-|g| is flushed to 0, sigma is 1 or
    0).  The band's edges are tight: each form fails just inside it."""
    bits = np.arange(65536, dtype=np.uint32)
    g = (bits << 16).view(np.float32)
    expo = (bits >> 7) & 0xFF
    with np.errstate(all="ignore"):
        got = S.silu_spec(g).view(np.uint32)
        tiny = (g * np.float32(0.5)).astype(np.float32).view(np.uint32)
        large = (g * np.where(g >= 0, np.float32(1.0), np.float32(0.0))).astype(np.float32)
    large = large.view(np.uint32)
    below, above = expo < 102, expo > 133
    assert np.array_equal(got[below], tiny[below])
    assert np.array_equal(got[above], large[above])
    assert not np.array_equal(got[expo == 102], tiny[expo == 102])
    assert not np.array_equal(got[expo == 133], large[expo == 133])


def test_swiglu_worked_blocks():
    for name, attrs, _, body in cases("swiglu_blocks.txt", 4):
        gate = np.array(body[0].split(), np.float32)
        up = np.array(body[1].split(), np.float32)
        y = np.empty(32, np.float32)
        y[0::2] = gate
        y[1::2] = up
        h = S.swiglu(y[None])
        q, sc = Q.nvfp4_quantize_blocks(h, np.float32(attrs["s"]))
        assert int(sc[0]) == int(body[2].split()[1], 16), name
        assert np.array_equal(q[0], np.array(body[3].split(), np.uint8)), name


def test_swiglu_mx_worked_blocks():
    """swiglu_quantize in the MX formats on one-row groups, against the
    hand-worked blocks (element codes before packing and the E8M0 code)."""
    for name, attrs, _, body in cases("swiglu_mx_blocks.txt", 4):
        fmt = attrs["fmt"]
        gate = np.array(body[0].split(), np.float32)
        up = np.array(body[1].split(), np.float32)
        y = np.empty((1, 64), np.float32)
        y[0, 0::2] = gate
        y[0, 1::2] = up
        ro = np.array([0, 1], np.uint32)
        so = np.array([0, 128], np.uint32)
        out, sf = S.swiglu_quantize(y, None, ro, so, np.array([0], np.int32), fmt=fmt)
        codes = np.array([int(c, 16) for c in body[3].split()], np.uint8)
        got = out[0] if fmt == "mxfp8" else F.unpack_e2m1(out[0:1])[0]
        assert np.array_equal(got, codes), name
        assert int(L.unswizzle(sf, 128, 1)[0, 0]) == int(body[2].split()[1], 16), name


def test_swiglu_gate_up_order():
    # gate = 1, up = 3  ->  silu(1) * 3;  swapping would give silu(3) * 1
    h = S.swiglu(np.array([[1.0, 3.0]], np.float32))[0, 0]
    assert abs(h - 3.0 / (1.0 + np.exp(-1.0))) < 1e-6


def test_swiglu_quantize_grouping():
    rng = np.random.default_rng(30)
    I = 64
    counts = [3, 0, 130]
    ro = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    so = Q.padded_scale_offsets(ro)
    ids = np.array([4, 0, 2], np.int32)
    T = int(ro[-1]) + 2
    y = F.round_bf16(rng.normal(0, 2, (T, 2 * I))).astype(np.float32)
    s = rng.uniform(0.002, 0.01, 8).astype(np.float32)
    out0 = np.full((T, I // 2), 0x77, np.uint8)
    out, sf = S.swiglu_quantize(y, s, ro, so, ids, out=out0)
    kv = I // 16
    lg = L.unswizzle(sf, int(so[-1]), kv)
    h = S.swiglu(y)
    for g, e in enumerate(ids):
        r0, r1, p0 = int(ro[g]), int(ro[g + 1]), int(so[g])
        q, sc = Q.quantize_rows("nvfp4", h[r0:r1], s[e])
        assert np.array_equal(out[r0:r1], q)
        assert np.array_equal(lg[p0:p0 + r1 - r0], sc)
        assert not lg[p0 + r1 - r0:int(so[g + 1])].any()
    assert np.all(out[int(ro[-1]):] == 0x77)
