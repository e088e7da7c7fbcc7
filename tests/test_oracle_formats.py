"""Pins of the oracle's element codecs and scale layout against values fixed
outside the oracle: the format tables, PyTorch's own float8 / bfloat16
conversions (library routines), brute-force searches, hand-worked offsets."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import layout as L
from tests._golden import lines


def test_e2m1_table_matches_format_definition():
    want = {}
    for s in lines("e2m1_codes.txt"):
        c, v = s.split()
        want[int(c)] = float(v)
    for c in range(16):
        got = F.e2m1_value(c)
        assert got == want[c] and np.signbit(got) == np.signbit(want[c]), c
    assert np.array_equal(F.decode_e2m1(np.arange(16)), [want[c] for c in range(16)])


def test_e2m1_roundtrip_all_codes():
    codes = np.arange(16, dtype=np.uint8)
    assert np.array_equal(F.encode_e2m1(F.decode_e2m1(codes)), codes)


def test_e2m1_rounding_cases():
    for s in lines("e2m1_rounding.txt"):
        x, c = s.split()
        assert int(F.encode_e2m1(np.float64(x))) == int(c), s


def test_e2m1_encode_is_nearest_brute_force():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.uniform(-8, 8, 20000),
                        np.arange(-800, 801) / 100.0])
    got = F.encode_e2m1(x).astype(np.int64)
    vals = np.array([F.e2m1_value(c) for c in range(16)])
    for xi, ci in zip(x, got):
        d = np.abs(vals - xi)
        d[np.signbit(vals) != np.signbit(xi)] = np.inf  # sign is kept
        best = np.flatnonzero(d == d.min())
        if len(best) > 1:
            best = [b for b in best if (b & 1) == 0]
        assert ci == best[0], (xi, ci, best)


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = F.decode_e4m3(np.arange(256))
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert nan.sum() == 2 and nan[0x7F] and nan[0xFF]
    assert np.array_equal(got[~nan], ref[~nan])
    assert F.e4m3_value(0x7E) == 448.0 and F.e4m3_value(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne():
    rng = np.random.default_rng(2)
    x = np.concatenate([
        rng.normal(0, 1, 20000), rng.normal(0, 100, 20000),
        rng.uniform(-448, 448, 20000), rng.uniform(-2e-3, 2e-3, 20000),
        # exact midpoints between neighbouring codes
        (F.E4M3_TABLE[1:0x7E] + F.E4M3_TABLE[2:0x7F]) / 2,
        -(F.E4M3_TABLE[1:0x7E] + F.E4M3_TABLE[2:0x7F]) / 2,
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = F.encode_e4m3(x)
    assert np.array_equal(got, ref)


def test_e4m3_saturation_and_underflow():
    assert int(F.encode_e4m3(500.0)) == 0x7E
    assert int(F.encode_e4m3(1e30)) == 0x7E
    assert int(F.encode_e4m3(-449.0)) == 0xFE
    assert int(F.encode_e4m3(2.0 ** -10)) == 0x00      # tie -> even code 0
    assert int(F.encode_e4m3(-(2.0 ** -10))) == 0x80
    assert int(F.encode_e4m3(2.0 ** -10 * 1.0001)) == 0x01


def test_e8m0_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = F.decode_e8m0(np.arange(256))
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])


def test_bf16_encode_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.normal(0, 1, 50000), rng.normal(0, 1e30, 1000),
        rng.normal(0, 1e-39, 1000),                 # fp32 subnormals
        np.array([0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8]),
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.encode_bf16(x), ref)


def test_bf16_roundtrip_all_finite():
    bits = np.arange(65536, dtype=np.uint32)
    v = F.decode_bf16(bits)
    fin = np.isfinite(v)
    assert np.array_equal(F.encode_bf16(v[fin]), bits[fin].astype(np.uint16))


def test_pack_low_nibble_first():
    assert F.pack_e2m1(np.array([1, 2], np.uint8))[0] == 0x21
    rng = np.random.default_rng(4)
    c = rng.integers(0, 16, (5, 64)).astype(np.uint8)
    assert np.array_equal(F.unpack_e2m1(F.pack_e2m1(c)), c)


def test_sf_layout_positions():
    for s in lines("sf_layout_positions.txt"):
        r, c, kv, off = map(int, s.split())
        assert int(L.sf_offset(r, c, kv)) == off, s


def test_sf_layout_is_a_bijection_and_roundtrips():
    rng = np.random.default_rng(5)
    for rows, kv in [(128, 4), (256, 8), (384, 6), (128, 96)]:
        rr, cc = np.meshgrid(np.arange(rows), np.arange(kv), indexing="ij")
        offs = L.sf_offset(rr, cc, kv).reshape(-1)
        assert len(np.unique(offs)) == offs.size
        assert offs.max() < L.physical_bytes(rows, kv)
        x = rng.integers(0, 256, (rows, kv)).astype(np.uint8)
        buf = L.swizzle(x)
        assert np.array_equal(L.unswizzle(buf, rows, kv), x)
        if kv % 4:
            mask = np.ones(buf.size, bool)
            mask[offs] = False
            assert not buf[mask].any()


def test_interleave_rows_hand_case():
    gate = np.array([[[1, 2], [3, 4]], [[9, 10], [11, 12]]], np.uint8)
    up = np.array([[[5, 6], [7, 8]], [[13, 14], [15, 16]]], np.uint8)
    want = np.array([[[1, 2], [5, 6], [3, 4], [7, 8]],
                     [[9, 10], [13, 14], [11, 12], [15, 16]]], np.uint8)
    assert np.array_equal(L.interleave_rows(gate, up), want)
