"""Pins of the oracle's exp / SiLU definition (against long-double exp and
limits fixed by the mathematics) and of the chained SwiGLU requantization
(hand-worked blocks, gate/up order, grouping)."""
import numpy as np

from oracle import formats as F
from oracle import layout as L
from oracle import quantize as Q
from oracle import swiglu as S
from tests._golden import cases


def test_exp_spec_accuracy_vs_long_double():
    x = np.concatenate([np.linspace(-87.0, 88.5, 400001),
                        F.decode_bf16(np.arange(0x0000, 0x42B0, 7)),
                        -F.decode_bf16(np.arange(0x0000, 0x42AE, 7))]).astype(np.float32)
    got = S.exp_spec(x).astype(np.longdouble)
    ref = np.exp(x.astype(np.longdouble))
    rel = np.abs(got - ref) / ref
    assert rel.max() <= 2.0 ** -21, float(rel.max())


def test_exp_spec_special_points():
    assert S.exp_spec(np.float32(0.0)) == 1.0
    assert np.isinf(S.exp_spec(np.float32(89.0)))
    assert np.isinf(S.exp_spec(np.float32(88.8)))          # overflows naturally
    assert np.isfinite(S.exp_spec(np.float32(88.7)))
    assert S.exp_spec(np.float32(-104.0)) == 0.0
    # subnormal results: within one subnormal step of the true value
    for x in (-90.0, -100.0, -103.0):
        got = float(S.exp_spec(np.float32(x)))
        assert abs(got - np.exp(x)) <= 2.0 ** -149


def test_silu_limits():
    assert S.silu_spec(np.float32(0.0)) == 0.0
    assert S.silu_spec(np.float32(32.0)) == 32.0
    assert S.silu_spec(np.float32(1000.0)) == 1000.0
    r = S.silu_spec(np.float32(-200.0))
    assert r == 0.0 and np.signbit(r)
    g = np.linspace(-60, 60, 20001).astype(np.float32)
    ref = g.astype(np.float64) / (1.0 + np.exp(-g.astype(np.float64)))
    got = S.silu_spec(g).astype(np.float64)
    big = np.abs(ref) > 1e-30
    assert np.max(np.abs(got[big] - ref[big]) / np.abs(ref[big])) < 2.0 ** -20


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
