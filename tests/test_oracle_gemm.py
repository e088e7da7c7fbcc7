"""Pins of the oracle's grouped GEMMs: hand-computed cases, exact rational
brute force on tiny ragged inputs, a dense special case through PyTorch's own
float8 decode, and invariants (empty groups, power-of-two scaling)."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import gemm as G
from oracle import layout as L
from tests._golden import lines


def _kv(name):
    out = {}
    for s in lines(name):
        k, *v = s.split()
        out[k] = v
    return out


def test_fp8_rowwise_hand_case():
    d = _kv("fp8_rowwise_2x2x16.txt")
    a_rows = [float(v) for v in d["a_row"]]
    b_rows = [float(v) for v in d["b_row"]]
    a = np.array([[F.encode_e4m3(v)] * 16 for v in a_rows], np.uint8)
    b = np.array([[[F.encode_e4m3(v)] * 16 for v in b_rows]], np.uint8)
    out = G.grouped_matmul_rowwise_fp8(
        a, b, np.array(d["a_scale"], np.float32), np.array([d["b_scale"]], np.float32),
        [0, 2], [0])
    assert np.array_equal(F.decode_bf16(out).reshape(-1), np.array(d["out"], np.float32))


def test_nvfp4_blockscaled_hand_case():
    d = _kv("nvfp4_gemm_2x2x32.txt")

    def row(key):
        v = d[key]
        elems = [float(v[0])] * 16 + [float(v[1])] * 16
        return F.encode_e2m1(np.array(elems)), F.encode_e4m3(np.array([float(v[3]), float(v[4])]))

    a_q, a_s = zip(*(row(k) for k in ("a0", "a1")))
    b_q, b_s = zip(*(row(k) for k in ("b0", "b1")))
    a = F.pack_e2m1(np.stack(a_q))
    b = F.pack_e2m1(np.stack(b_q))[None]
    a_log = np.zeros((128, 2), np.uint8)
    a_log[:2] = np.stack(a_s)
    b_log = np.zeros((128, 2), np.uint8)
    b_log[:2] = np.stack(b_s)
    out = G.grouped_matmul_blockscaled(
        "nvfp4", a, L.swizzle(a_log), b, L.swizzle(b_log),
        np.array([float(d["expert_scale"][0])], np.float32),
        [0, 2], [0, 128], [0], N=2, K=32, scale_rows_total=128)
    assert np.array_equal(F.decode_bf16(out).reshape(-1), np.array(d["out"], np.float32))


def _ragged(rng, counts, E):
    ro = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    ids = rng.permutation(E)[: len(counts)].astype(np.int32)
    return ro, ids


def test_fp8_rowwise_brute_force_exact():
    rng = np.random.default_rng(20)
    E, N, K = 3, 5, 32
    counts = [4, 0, 6]
    ro, ids = _ragged(rng, counts, E)
    T = int(ro[-1]) + 2
    a = rng.integers(0, 256, (T, K)).astype(np.uint8)
    b = rng.integers(0, 256, (E, N, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x3C
    b[(b & 0x7F) == 0x7F] = 0x41
    sa = rng.uniform(0.01, 0.1, T).astype(np.float32)
    sb = rng.uniform(0.005, 0.05, (E, N)).astype(np.float32)
    canary = np.full((T, N), 0xBEEF, np.uint16)
    out = G.grouped_matmul_rowwise_fp8(a, b, sa, sb, ro, ids, out=canary)
    written = np.zeros(T, bool)
    for g in range(len(counts)):
        e = int(ids[g])
        for t in range(int(ro[g]), int(ro[g + 1])):
            written[t] = True
            for n in range(N):
                acc = sum(Fraction(F.e4m3_value(a[t, k])) * Fraction(F.e4m3_value(b[e, n, k]))
                          for k in range(K))
                exact = acc * Fraction(float(sa[t])) * Fraction(float(sb[e, n]))
                assert out[t, n] == F.encode_bf16(float(exact)), (t, n)
    assert np.all(out[~written] == 0xBEEF)


@pytest.mark.parametrize("fmt,with_rows", [("nvfp4", False), ("nvfp4", True), ("mxfp8", False),
                                           ("mxfp4", False)])
def test_blockscaled_brute_force_exact(fmt, with_rows):
    rng = np.random.default_rng(21)
    v = 16 if fmt == "nvfp4" else 32
    E, N, K = 3, 4, 64
    kv = K // v
    counts = [3, 0, 5]
    ro, ids = _ragged(rng, counts, E)
    so = np.array([0, 128, 128, 256], np.uint32)
    T = int(ro[-1]) + 1
    rows = 256
    if fmt == "mxfp8":
        a = rng.integers(0, 256, (T, K)).astype(np.uint8)
        b = rng.integers(0, 256, (E, N, K)).astype(np.uint8)
        a[(a & 0x7F) == 0x7F] = 0x3C
        b[(b & 0x7F) == 0x7F] = 0x41
        ev = F.e4m3_value
        unpacked_a, unpacked_b = a, b
    else:
        a = rng.integers(0, 256, (T, K // 2)).astype(np.uint8)
        b = rng.integers(0, 256, (E, N, K // 2)).astype(np.uint8)
        ev = F.e2m1_value
        unpacked_a, unpacked_b = F.unpack_e2m1(a), F.unpack_e2m1(b)
    if fmt == "nvfp4":
        sa_log = rng.integers(0x20, 0x48, (rows, kv)).astype(np.uint8)
        sb_log = rng.integers(0x20, 0x48, (E, 128, kv)).astype(np.uint8)
        sv = F.e4m3_value
        es = rng.uniform(0.5, 2, E).astype(np.float32)
    else:
        sa_log = rng.integers(120, 135, (rows, kv)).astype(np.uint8)
        sb_log = rng.integers(120, 135, (E, 128, kv)).astype(np.uint8)
        sv = F.e8m0_value
        es = None
    a_sf = L.swizzle(sa_log)
    b_sf = np.concatenate([L.swizzle(sb_log[e]) for e in range(E)])
    # optional per-row scales (bf16 values): multiply in with the expert scale
    rs = F.round_bf16(rng.uniform(0.5, 2.0, T)).astype(np.float64) if with_rows else None
    out = G.grouped_matmul_blockscaled(fmt, a, a_sf, b, b_sf, es, ro, so, ids,
                                       N=N, K=K, scale_rows_total=rows, row_scales=rs)
    for g in range(len(counts)):
        e = int(ids[g])
        for i, t in enumerate(range(int(ro[g]), int(ro[g + 1]))):
            p = int(so[g]) + i
            for n in range(N):
                acc = sum(Fraction(ev(unpacked_a[t, k])) * Fraction(sv(sa_log[p, k // v]))
                          * Fraction(ev(unpacked_b[e, n, k])) * Fraction(sv(sb_log[e, n, k // v]))
                          for k in range(K))
                if es is not None:
                    acc *= Fraction(float(es[e]))
                if rs is not None:
                    acc *= Fraction(float(rs[t]))
                assert out[t, n] == F.encode_bf16(float(acc)), (t, n)


def test_fp8_rowwise_dense_case_matches_torch():
    """G = 1, E = 1 is a dense rowwise-scaled GEMM; decode through PyTorch."""
    g = torch.Generator().manual_seed(0)
    a = (torch.randn(40, 64, generator=g)).to(torch.float8_e4m3fn)
    b = (torch.randn(1, 24, 64, generator=g) * 0.5).to(torch.float8_e4m3fn)
    sa = torch.rand(40, generator=g) * 0.1
    sb = torch.rand(1, 24, generator=g) * 0.05
    ref = (a.double() @ b[0].double().T) * sa.double()[:, None] * sb.double()
    _, f64 = G.grouped_matmul_rowwise_fp8(a.view(torch.uint8).numpy(), b.view(torch.uint8).numpy(),
                                          sa.numpy(), sb.numpy(), [0, 40], [0], return_f64=True)
    assert np.allclose(f64, ref.numpy(), rtol=1e-12, atol=0)


def test_fp8_rowwise_power_of_two_scaling_is_exact():
    rng = np.random.default_rng(22)
    a = rng.integers(0, 0x7E, (16, 32)).astype(np.uint8)
    b = rng.integers(0, 0x7E, (2, 8, 32)).astype(np.uint8)
    sa = rng.uniform(0.01, 0.1, 16).astype(np.float32)
    sb = rng.uniform(0.01, 0.1, (2, 8)).astype(np.float32)
    o1 = G.grouped_matmul_rowwise_fp8(a, b, sa, sb, [0, 9, 16], [1, 0])
    o2 = G.grouped_matmul_rowwise_fp8(a, b, sa * 2, sb, [0, 9, 16], [1, 0])
    assert np.array_equal(F.decode_bf16(o1) * 2, F.decode_bf16(o2))
