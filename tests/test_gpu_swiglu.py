"""GPU parity of the SwiGLU + NVFP4 requantization, through the C ABI:
* the chained kernel (bf16 y -> packed + scales) is bit-exact against the
  oracle on generator-made y (small ragged cases, special values, and the
  131072-row workload on sampled rows);
* the fused GEMM + SwiGLU + requant writes exactly the bytes of the chained
  path (block-scaled GEMM to bf16, then the chained kernel), whole buffers,
  on small ragged cases and the full 128-expert workload."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import moeq, synth
from oracle import layout as L
from oracle import quantize as Q
from oracle import swiglu as S
from tests._util import (DEV, group_sample_rows, groups_from_counts, need_gpu, to_dev_i32,
                         to_dev_u32, u8)
from tests.test_gpu_gemm import blockscaled_inputs

pytestmark = pytest.mark.gpu


def _run_chained_swiglu(y, ots, ro, so, ids, E, rows):
    T, I2 = y.shape
    I = I2 // 2
    out = torch.full((T, I // 2), 0xA5, dtype=torch.uint8, device=DEV)
    sf = torch.full((moeq.sf_bytes(rows, I // 16),), 0x5A, dtype=torch.uint8, device=DEV)
    moeq.swiglu_quantize(out, sf, y.to(DEV), ots.to(DEV), to_dev_u32(ro), to_dev_u32(so),
                         to_dev_i32(ids), E, rows)
    torch.cuda.synchronize()
    return u8(out), u8(sf)


@pytest.mark.parametrize("I", [64, 192, 576, 1536])
def test_swiglu_quantize_bit_exact(I):
    need_gpu()
    counts = [0, 1, 127, 128, 129, 40]
    ids = np.array([3, 1, 0, 4, 2, 5], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    so = Q.padded_scale_offsets(ro)
    T = int(ro[-1]) + 4
    rows = int(so[-1]) + 128
    y = synth.bf16_normal((T, 2 * I), 2.0, seed=I, outlier_p=0.01, outlier_scale=40.0)
    yv = y.view(torch.int16)
    yv[0, :16] = torch.tensor(np.float32([40.0, -3, -40, 2, 100, 1, -100, 1, 0, 0, -0.0, 5, 5,
                                          -0.0, 1e-30, 1]).astype(np.float32)).to(
        torch.bfloat16).view(torch.int16)
    ots = synth.uniform((6,), 0.001, 0.004, seed=I + 1)
    out, sf = _run_chained_swiglu(y, ots, ro, so, ids, 6, rows)
    want_out, want_sf = S.swiglu_quantize(
        y.float().numpy(), ots.numpy(), ro, so, ids,
        out=np.full((T, I // 2), 0xA5, np.uint8),
        scales=np.full(L.physical_bytes(rows, I // 16), 0x5A, np.uint8), scale_rows_total=rows)
    assert np.array_equal(out, want_out)
    assert np.array_equal(sf, want_sf)


@pytest.mark.parametrize("I", [576, 1536])
def test_swiglu_quantize_y_16_byte_aligned(I):
    """y starting 16 bytes past a 32-byte boundary (the kernel then reads
    each lane's 64 bytes as four 16-byte loads) gives the bytes of the
    32-byte aligned call; both equal the oracle's."""
    need_gpu()
    counts = [5, 0, 130, 1, 64]
    ids = np.array([2, 0, 1, 4, 3], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    so = Q.padded_scale_offsets(ro)
    T, rows = int(ro[-1]), int(so[-1])
    y = synth.bf16_normal((T, 2 * I), 2.0, seed=I + 5, outlier_p=0.01, outlier_scale=30.0)
    ots = synth.uniform((5,), 0.001, 0.004, seed=I + 6)
    base = torch.zeros(T * 2 * I + 64, dtype=torch.bfloat16, device=DEV)
    off = (-base.data_ptr() // 2) % 16 + 8  # 16 bytes past a 32-byte boundary
    y_off = base[off:off + T * 2 * I].view(T, 2 * I)
    y_off.copy_(y.to(DEV))
    assert y_off.data_ptr() % 32 == 16
    out_a, sf_a = _run_chained_swiglu(y, ots, ro, so, ids, 5, rows)
    out_u, sf_u = _run_chained_swiglu(y_off, ots, ro, so, ids, 5, rows)
    assert np.array_equal(out_a, out_u) and np.array_equal(sf_a, sf_u)
    want_out, want_sf = S.swiglu_quantize(
        y.float().numpy(), ots.numpy(), ro, so, ids,
        out=np.full((T, I // 2), 0xA5, np.uint8),
        scales=np.full(L.physical_bytes(rows, I // 16), 0x5A, np.uint8), scale_rows_total=rows)
    assert np.array_equal(out_a, want_out)
    assert np.array_equal(sf_a, want_sf)


def test_swiglu_quantize_full_size_sampled():
    """131072 rows over 128 experts, I = 1536, on sampled rows."""
    need_gpu()
    counts = synth.routing_counts(16384, 8, 128, seed=0)
    ro, ids = synth.ragged_groups(counts)
    so = Q.padded_scale_offsets(ro)
    T, I, rows = int(ro[-1]), 1536, int(so[-1])
    y = synth.bf16_normal((T, 2 * I), 3.0, seed=60, device=DEV)
    ots = synth.uniform((128,), 0.002, 0.01, seed=61)
    out, sf = _run_chained_swiglu(y, ots, ro, so, ids, 128, rows)
    # every group: its first, last and middle rows and one row per 128-row block
    sel = np.concatenate(group_sample_rows(ro))
    grp = np.searchsorted(ro, sel, side="right") - 1
    ysel = y[torch.from_numpy(sel).to(DEV)].float().cpu().numpy()
    lg = L.unswizzle(sf, rows, I // 16)
    h = S.swiglu(ysel)
    for g in np.unique(grp):
        m = grp == g
        q, sc = Q.quantize_rows("nvfp4", h[m], ots.numpy()[ids[g]])
        assert np.array_equal(out[sel[m]], q)
        assert np.array_equal(lg[int(so[g]) + sel[m] - int(ro[g])], sc)
    for g in range(len(ids)):
        r = int(ro[g + 1] - ro[g])
        assert not lg[int(so[g]) + r:int(so[g + 1])].any()


def _fused_and_chained(a, asf, b, bsf, es, ots, ro, so, ids, I, K, rows):
    T = a.shape[0]
    N = 2 * I
    dev = lambda t: t.to(DEV)
    # chained: block-scaled GEMM -> bf16 y -> SwiGLU + NVFP4
    y = torch.full((T, N), 0.0, dtype=torch.bfloat16, device=DEV)
    moeq.grouped_matmul_blockscaled("nvfp4", y, dev(a), dev(asf), dev(b), dev(bsf), dev(es),
                                    to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids), N, K, rows)
    c1 = torch.full((T, I // 2), 0xA5, dtype=torch.uint8, device=DEV)
    s1 = torch.full((moeq.sf_bytes(rows, I // 16),), 0x5A, dtype=torch.uint8, device=DEV)
    moeq.swiglu_quantize(c1, s1, y, dev(ots), to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids),
                         b.shape[0], rows)
    # fused
    c2 = torch.full_like(c1, 0xA5)
    s2 = torch.full_like(s1, 0x5A)
    moeq.grouped_matmul_swiglu(c2, s2, dev(a), dev(asf), dev(b), dev(bsf), dev(es), dev(ots),
                               to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids), I, K, rows)
    torch.cuda.synchronize()
    return c1, s1, c2, s2


@pytest.mark.parametrize("I,K", [(64, 256), (192, 512), (256, 1024)])
def test_fused_equals_chained_small(I, K):
    need_gpu()
    counts = [0, 1, 127, 129, 260, 3]
    ids = np.array([4, 0, 2, 5, 1, 3], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    so = Q.padded_scale_offsets(ro)
    rows = int(so[-1]) + 128
    T = int(ro[-1]) + 5
    a, asf, b, bsf, es = blockscaled_inputs("nvfp4", T, 6, 2 * I, K, rows, seed=I + K)
    ots = synth.uniform((6,), 0.05, 0.2, seed=3)
    c1, s1, c2, s2 = _fused_and_chained(a, asf, b, bsf, es, ots, ro, so, ids, I, K, rows)
    assert torch.equal(c1, c2)
    assert torch.equal(s1, s2)
    # and the output is not trivial
    assert (c1[:int(ro[-1])] != 0).float().mean() > 0.3


@pytest.mark.parametrize("empty_groups", [0, 507])
def test_fused_equals_chained_extreme_scales(empty_groups):
    """Expert scales that push the bf16 gates below the SiLU table's band
    (1e-36: subnormal and tiny gates), into it (1), above it (1e4: |g| >=
    128) and past the bf16 range (1e38: +-inf gates, NaN from -inf * 0), and
    zero: the fused kernel's table lookups and closed forms give the chained
    kernel's bytes."""
    need_gpu()
    I, K = 128, 256
    # 507 empty groups appended make 513: a launch past the table kernel's
    # 512 groups, which computes the SiLU
    counts = [130, 7, 129, 64, 1, 200] + [0] * empty_groups
    ids = np.array([0, 1, 2, 3, 4, 5] + [g % 6 for g in range(empty_groups)], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    so = Q.padded_scale_offsets(ro)
    rows = int(so[-1])
    T = int(ro[-1])
    a, asf, b, bsf, _ = blockscaled_inputs("nvfp4", T, 6, 2 * I, K, rows, seed=41)
    es = torch.tensor([1e-36, 1.0, 1e4, 1e38, 0.0, 3e-8], dtype=torch.float32)
    ots = torch.tensor([1.0, 0.1, 1e3, 1.0, 1.0, 1e-6], dtype=torch.float32)
    c1, s1, c2, s2 = _fused_and_chained(a, asf, b, bsf, es, ots, ro, so, ids, I, K, rows)
    assert torch.equal(c1, c2)
    assert torch.equal(s1, s2)
    # the cases occurred: infinite gates, gates below the band, gates above it
    y = torch.zeros((T, 2 * I), dtype=torch.bfloat16, device=DEV)
    moeq.grouped_matmul_blockscaled("nvfp4", y, a.to(DEV), asf.to(DEV), b.to(DEV), bsf.to(DEV),
                                    es.to(DEV), to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids),
                                    2 * I, K, rows)
    g = y[:, 0::2].float().cpu()
    assert torch.isinf(g).any() and (g == float("-inf")).any()
    assert ((g != 0) & (g.abs() < 2.0 ** -25)).any()
    assert (g.abs() >= 128).any() and torch.isfinite(g[(g.abs() >= 128)]).any()


def test_fused_equals_chained_full_size():
    """128 experts, 131072 rows, K = 4096, I = 1536: whole buffers equal."""
    need_gpu()
    counts = synth.routing_counts(16384, 8, 128, seed=0)
    ro, ids = synth.ragged_groups(counts)
    so = Q.padded_scale_offsets(ro)
    T, I, K, rows = int(ro[-1]), 1536, 4096, int(so[-1])
    a, asf, b, bsf, es = blockscaled_inputs("nvfp4", T, 128, 2 * I, K, rows, seed=70, device=DEV)
    ots = synth.uniform((128,), 1.0, 4.0, seed=71, device=DEV)
    c1, s1, c2, s2 = _fused_and_chained(a, asf, b, bsf, es, ots, ro, so, ids, I, K, rows)
    assert torch.equal(c1, c2)
    assert torch.equal(s1, s2)
    codes = u8(s1)
    assert (codes != 0).mean() > 0.5 and (codes < 0x7E).mean() > 0.5


def test_fused_missing_scales_is_invalid_arg():
    need_gpu()
    z = torch.zeros(16, dtype=torch.uint8, device=DEV)
    o = torch.zeros(2, dtype=torch.int32, device=DEV)
    e = torch.zeros(1, dtype=torch.int32, device=DEV)
    b = torch.zeros((1, 128, 128), dtype=torch.uint8, device=DEV)
    with pytest.raises(moeq.MoeqError) as ex:
        moeq.grouped_matmul_swiglu(z, z, torch.zeros((1, 128), dtype=torch.uint8, device=DEV), z,
                                   b, z, None, torch.ones(1, device=DEV), o, o, e, 64, 256, 128)
    assert ex.value.status == 1
