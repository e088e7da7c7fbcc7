"""Pins of the oracle's quantizers: hand-worked blocks, brute-force optimality
of every chosen code, properties fixed by the scale rules, and the grouping
semantics (padding rows zero, rows outside groups untouched, permutation)."""
import numpy as np
import pytest

from oracle import formats as F
from oracle import layout as L
from oracle import quantize as Q
from tests._golden import cases


def test_nvfp4_worked_blocks():
    for name, attrs, _, body in cases("nvfp4_blocks.txt", 3):
        x = np.array(body[0].split(), dtype=np.float32)
        want_scale = int(body[1].split()[1], 16)
        want_codes = np.array(body[2].split(), dtype=np.uint8)
        q, sc = Q.nvfp4_quantize_blocks(x[None, :], np.float32(attrs["s"]))
        assert int(sc[0]) == want_scale, name
        assert np.array_equal(q[0], want_codes), name


def test_mx_worked_blocks():
    for name, _, flags, body in cases("mx_blocks.txt", 3):
        fmt = flags[0]
        x = np.zeros(32, np.float64)
        for item in body[0].split()[1:]:
            i, v = item.split(":")
            x[int(i)] = float(v)
        want_c = int(body[1].split()[1])
        want_q = np.zeros(32, np.uint8)
        for item in body[2].split()[1:]:
            i, v = item.split(":")
            want_q[int(i)] = int(v, 16)
        q, c = Q.mx_quantize_blocks(x[None, :], "e4m3" if fmt == "mxfp8" else "e2m1")
        assert int(c[0]) == want_c, name
        assert np.array_equal(q[0], want_q), name


def _blocks(rng, n, v):
    x = rng.normal(0, 1, (n, v)) * np.exp(rng.uniform(-6, 6, (n, 1)))
    x[rng.random((n, v)) < 0.02] *= 50
    return F.round_bf16(x).astype(np.float32)


def test_nvfp4_codes_are_nearest_and_scale_direction():
    rng = np.random.default_rng(10)
    x = _blocks(rng, 1000, 16)
    s = np.float32(0.013)
    q, sc = Q.nvfp4_quantize_blocks(x, s)
    sb = F.decode_e4m3(sc)
    assert np.all(sb <= 448) and np.all(F.decode_e2m1(q) <= 6)
    # The scale code is the E4M3 value nearest to amax / (6 s), up to the
    # fp32 rounding of that quotient (brute force over all finite codes).
    target = np.abs(x).max(1).astype(np.float64) / (6.0 * np.float64(s))
    fin = np.isfinite(F.E4M3_TABLE) & (np.arange(256) < 0x80)
    table = F.E4M3_TABLE[fin]
    for t, c in zip(target, sc):
        d = np.abs(table - t)
        assert abs(F.e4m3_value(c) - t) <= d.min() * (1 + 1e-6) + 1e-12 or t > 448
    # Every element code is the E2M1 value nearest to x * (1/s) / sb.
    vals = F.E2M1_TABLE
    for i in range(0, 1000, 7):
        if sb[i] == 0:
            assert not q[i].any()
            continue
        r = np.float32(np.float32(1) / s) / np.float32(sb[i])
        for xv, qc in zip(x[i], q[i]):
            y = float(np.float32(xv * np.float32(r)))
            d = np.abs(vals - y)
            d[np.signbit(vals) != np.signbit(y)] = np.inf
            assert d[qc] == d.min()
    # Blocks whose scale is a normal, unsaturated E4M3 number map their
    # largest element to magnitude 6: the scale is amax/6 in element units.
    ok = (target >= 2.0 ** -6) & (target <= 440)
    amax_code = np.take_along_axis(q, np.abs(x).argmax(1)[:, None], 1)[:, 0] & 7
    assert ok.sum() > 500 and np.all(amax_code[ok] == 7)


@pytest.mark.parametrize("elem,emax,elem_max", [("e4m3", 8, 448.0), ("e2m1", 2, 6.0)])
def test_mx_floor_rule_and_nearest(elem, emax, elem_max):
    rng = np.random.default_rng(11)
    x = _blocks(rng, 500, 32).astype(np.float64)
    q, c = Q.mx_quantize_blocks(x, elem)
    m = np.abs(x).max(1)
    c = c.astype(np.int64)
    # floor rule: 2^(c-127+emax) <= amax < 2^(c-127+emax+1)
    assert np.all(2.0 ** (c - 127 + emax) <= m) and np.all(m < 2.0 ** (c - 127 + emax + 1))
    dec = F.decode_e4m3 if elem == "e4m3" else F.decode_e2m1
    table = F.E4M3_TABLE[:0x7F] if elem == "e4m3" else F.E2M1_TABLE[:8]
    y = x * 2.0 ** (127 - c)[:, None]
    got = np.abs(dec(q))
    # nearest finite magnitude (brute force), saturating at the format max
    d = np.abs(np.abs(y)[..., None] - table[None, None, :])
    assert np.all(np.abs(got - np.abs(y)) <= d.min(-1) + 1e-300)
    assert np.all(got <= elem_max)
    assert np.array_equal(np.signbit(dec(q)), np.signbit(y))


def test_tensor_scale_from_amax():
    s = Q.tensor_scale_from_amax(np.array([2688.0, 0.0, 1.0], np.float32))
    assert s[0] == 1.0 and s[1] == 1.0 and s[2] == np.float32(1.0) / np.float32(2688.0)


def test_padded_scale_offsets():
    assert list(Q.padded_scale_offsets([0, 7, 23, 32])) == [0, 128, 256, 384]
    assert list(Q.padded_scale_offsets([0, 0, 129, 257])) == [0, 0, 256, 384]


def _grouped_case(rng, fmt, counts, ids, K=128):
    ro = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    so = Q.padded_scale_offsets(ro)
    T = int(ro[-1]) + 3                       # 3 trailing rows in no group
    x = F.round_bf16(rng.normal(0, 1, (T, K))).astype(np.float32)
    ts = Q.tensor_scale_from_amax(Q.group_amax(x, ro, ids, 8))
    rows = int(so[-1]) + 128                  # one extra 128-row block
    v = Q.block_size(fmt)
    ob = K if fmt == "mxfp8" else K // 2
    out0 = np.full((T, ob), 0xA5, np.uint8)
    sf0 = np.full(L.physical_bytes(rows, K // v), 0x5A, np.uint8)
    out, sf = Q.grouped_quantize(fmt, x, ro, so, ids, ts, out0, sf0, rows)
    return x, ro, so, ts, out0, sf0, out, sf, rows


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8", "mxfp4"])
def test_grouped_quantize_semantics(fmt):
    rng = np.random.default_rng(12)
    counts = [5, 0, 130, 1]
    ids = np.array([3, 1, 0, 6], np.int32)
    x, ro, so, ts, out0, sf0, out, sf, rows = _grouped_case(rng, fmt, counts, ids)
    K = x.shape[1]
    kv = K // Q.block_size(fmt)
    # rows in no group keep their bytes
    assert np.array_equal(out[int(ro[-1]):], out0[int(ro[-1]):])
    logical = L.unswizzle(sf, rows, kv)
    # scale rows at or past scales_offsets[G] keep their bytes
    assert np.all(logical[int(so[-1]):] == 0x5A)
    for g, e in enumerate(ids):
        r0, r1, p0, p1 = int(ro[g]), int(ro[g + 1]), int(so[g]), int(so[g + 1])
        q, sc = Q.quantize_rows(fmt, x[r0:r1], ts[e] if fmt == "nvfp4" else None)
        assert np.array_equal(out[r0:r1], q)
        assert np.array_equal(logical[p0:p0 + (r1 - r0)], sc)
        padded = (r1 - r0 + 127) // 128 * 128
        assert not logical[p0 + (r1 - r0):p0 + padded].any()  # padding rows zero
        assert np.all(logical[p0 + padded:p1] == 0x5A)       # slack rows untouched


def test_grouped_quantize_slack_scale_rows_untouched():
    """Offsets with more than the tight padding: only ceil128(r_g) rows of a
    group's scale range are written."""
    rng = np.random.default_rng(14)
    x = F.round_bf16(rng.normal(0, 1, (10, 128))).astype(np.float32)
    ro = np.array([0, 3, 10], np.uint32)
    so = np.array([0, 256, 512], np.uint32)
    sf0 = np.full(L.physical_bytes(512, 8), 0x5A, np.uint8)
    _, sf = Q.grouped_quantize("nvfp4", x, ro, so, np.array([0, 1], np.int32),
                               np.ones(2, np.float32), scales=sf0, scale_rows_total=512)
    lg = L.unswizzle(sf, 512, 8)
    assert not lg[3:128].any() and np.all(lg[128:256] == 0x5A)
    assert not lg[263:384].any() and np.all(lg[384:512] == 0x5A)


def test_grouped_quantize_group_permutation():
    """Permuting the groups (rows, padded scale rows and expert ids together)
    permutes the outputs and nothing else."""
    rng = np.random.default_rng(13)
    counts = [40, 3, 129]
    ids = np.array([2, 5, 1], np.int32)
    x, ro, so, ts, _, _, out, sf, rows = _grouped_case(rng, "nvfp4", counts, ids)
    perm = [2, 0, 1]
    counts_p = [counts[i] for i in perm]
    ro_p = np.concatenate([[0], np.cumsum(counts_p)]).astype(np.uint32)
    so_p = Q.padded_scale_offsets(ro_p)
    xp = np.concatenate([x[int(ro[i]):int(ro[i + 1])] for i in perm] + [x[int(ro[-1]):]])
    outp, sfp = Q.grouped_quantize("nvfp4", xp, ro_p, so_p, ids[perm], ts, scale_rows_total=rows)
    kv = x.shape[1] // 16
    lg = L.unswizzle(sf, rows, kv)
    lgp = L.unswizzle(sfp, rows, kv)
    for j, i in enumerate(perm):
        assert np.array_equal(outp[int(ro_p[j]):int(ro_p[j + 1])], out[int(ro[i]):int(ro[i + 1])])
        n = int(so[i + 1] - so[i])
        assert np.array_equal(lgp[int(so_p[j]):int(so_p[j]) + n], lg[int(so[i]):int(so[i]) + n])


def test_gather_rows_hand_case():
    # routing positions token * top_k + slot with top_k = 2: positions 5, 2,
    # 7, 0 belong to tokens 2, 1, 3, 0
    x = np.arange(4 * 3, dtype=np.float32).reshape(4, 3)
    got = Q.gather_rows(x, [5, 2, 7, 0], 2)
    assert np.array_equal(got, x[[2, 1, 3, 0]])
    assert np.array_equal(Q.gather_rows(x, [3, 1], 1), x[[3, 1]])


def test_group_amax():
    x = np.zeros((6, 16), np.float32)
    x[0, 3] = -7
    x[4, 1] = 2
    x[5, 0] = 9                               # row in no group
    amax = Q.group_amax(x, [0, 2, 2, 5], np.array([1, 0, 3]), 4)
    assert list(amax) == [0.0, 7.0, 0.0, 2.0]
