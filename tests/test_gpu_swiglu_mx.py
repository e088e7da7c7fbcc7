"""GPU parity of the MX SwiGLU requantization and of the per-row scales of
the fused NVFP4 kernel, through the C ABI:
* the chained SwiGLU + MXFP4 / MXFP8 kernel is bit-exact against the oracle
  (MX block rule on the fp32 SiLU outputs) on generator-made y;
* the fused MX GEMM + SwiGLU + MX requant writes exactly the bytes of the
  chained path (MX block-scaled GEMM to bf16, then the chained kernel);
* a_row_scales: all ones change nothing; powers of two per row equal the
  chained path on the exactly rescaled bf16 y; general bf16 row scales agree
  with the oracle pipeline (float64 GEMM, one bf16 rounding) up to the
  rounding differences of the fp32 accumulation."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import moeq, synth
from oracle import formats as F
from oracle import gemm as GM
from oracle import layout as L
from oracle import quantize as Q
from oracle import swiglu as S
from tests._util import DEV, groups_from_counts, need_gpu, to_dev_i32, to_dev_u32, u8
from tests.test_gpu_gemm import blockscaled_inputs

pytestmark = pytest.mark.gpu


def _ob(fmt, I):
    return I if fmt == "mxfp8" else I // 2


def _chained_mx(fmt, y, ro_d, so_d, ids_d, E, rows):
    T, I = y.shape[0], y.shape[1] // 2
    out = torch.full((T, _ob(fmt, I)), 0xA5, dtype=torch.uint8, device=DEV)
    sf = torch.full((moeq.sf_bytes(rows, I // 32),), 0x5A, dtype=torch.uint8, device=DEV)
    moeq.swiglu_quantize_mx(fmt, out, sf, y, ro_d, so_d, ids_d, E, rows)
    torch.cuda.synchronize()
    return out, sf


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("I", [128, 384, 640, 1536])
def test_swiglu_quantize_mx_bit_exact(fmt, I):
    need_gpu()
    counts = [0, 1, 127, 128, 129, 40]
    ids = np.array([3, 1, 0, 4, 2, 5], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    so = Q.padded_scale_offsets(ro)
    T = int(ro[-1]) + 4
    rows = int(so[-1]) + 128
    y = synth.bf16_normal((T, 2 * I), 2.0, seed=I + 7, outlier_p=0.01, outlier_scale=40.0)
    yv = y.view(torch.int16)
    # a row with special values, an all-zero block, and a block of tiny values
    yv[0, :16] = torch.tensor(np.float32([40.0, -3, -40, 2, 100, 1, -100, 1, 0, 0, -0.0, 5, 5,
                                          -0.0, 1e-30, 1])).to(torch.bfloat16).view(torch.int16)
    y[1, :64] = 0.0
    y[2, :64] = 1e-30
    out, sf = _chained_mx(fmt, y.to(DEV), to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids), 6,
                          rows)
    want_out, want_sf = S.swiglu_quantize(
        y.float().numpy(), None, ro, so, ids, fmt=fmt,
        out=np.full((T, _ob(fmt, I)), 0xA5, np.uint8),
        scales=np.full(L.physical_bytes(rows, I // 32), 0x5A, np.uint8), scale_rows_total=rows)
    assert np.array_equal(u8(out), want_out)
    assert np.array_equal(u8(sf), want_sf)


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
def test_swiglu_quantize_mx_y_16_byte_aligned(fmt):
    """y starting 16 bytes past a 32-byte boundary (16-byte loads) gives the
    bytes of the 32-byte aligned call."""
    need_gpu()
    I = 640
    ro, ids = groups_from_counts([5, 0, 130, 1, 64], [2, 0, 1, 4, 3])
    so = Q.padded_scale_offsets(ro)
    T, rows = int(ro[-1]), int(so[-1])
    y = synth.bf16_normal((T, 2 * I), 2.0, seed=31, device=DEV)
    base = torch.zeros(T * 2 * I + 64, dtype=torch.bfloat16, device=DEV)
    off = (-base.data_ptr() // 2) % 16 + 8  # 16 bytes past a 32-byte boundary
    y_off = base[off:off + T * 2 * I].view(T, 2 * I)
    y_off.copy_(y)
    assert y_off.data_ptr() % 32 == 16
    ro_d, so_d, ids_d = to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids)
    out_a, sf_a = _chained_mx(fmt, y, ro_d, so_d, ids_d, 5, rows)
    out_u, sf_u = _chained_mx(fmt, y_off, ro_d, so_d, ids_d, 5, rows)
    assert torch.equal(out_a, out_u) and torch.equal(sf_a, sf_u)


def _fused_and_chained_mx(fmt, a, asf, b, bsf, es, ro, so, ids, I, K, rows):
    T, N = a.shape[0], 2 * I
    dev = lambda t: None if t is None else t.to(DEV)
    ro_d, so_d, ids_d = to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids)
    y = torch.zeros((T, N), dtype=torch.bfloat16, device=DEV)
    moeq.grouped_matmul_blockscaled(fmt, y, dev(a), dev(asf), dev(b), dev(bsf), dev(es), ro_d,
                                    so_d, ids_d, N, K, rows)
    c1, s1 = _chained_mx(fmt, y, ro_d, so_d, ids_d, b.shape[0], rows)
    c2 = torch.full_like(c1, 0xA5)
    s2 = torch.full_like(s1, 0x5A)
    moeq.grouped_matmul_swiglu_mx(fmt, c2, s2, dev(a), dev(asf), dev(b), dev(bsf), dev(es),
                                  ro_d, so_d, ids_d, I, K, rows)
    torch.cuda.synchronize()
    return c1, s1, c2, s2


@pytest.mark.parametrize("fmt", ["mxfp8", "mxfp4"])
@pytest.mark.parametrize("I,K", [(128, 256), (384, 512), (256, 1024)])
@pytest.mark.parametrize("with_es", [True, False])
def test_fused_mx_equals_chained(fmt, I, K, with_es):
    need_gpu()
    counts = [0, 1, 127, 129, 260, 3]
    ids = np.array([4, 0, 2, 5, 1, 3], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    so = Q.padded_scale_offsets(ro)
    rows = int(so[-1]) + 128
    T = int(ro[-1]) + 5
    a, asf, b, bsf, es = blockscaled_inputs(fmt, T, 6, 2 * I, K, rows, seed=I + K + 3)
    c1, s1, c2, s2 = _fused_and_chained_mx(fmt, a, asf, b, bsf, es if with_es else None, ro, so,
                                           ids, I, K, rows)
    assert torch.equal(c1, c2)
    assert torch.equal(s1, s2)
    assert (c1[:int(ro[-1])] != 0).float().mean() > 0.3
    assert moeq.get_device_error() == 0


@pytest.mark.parametrize("empty_groups", [0, 507])
def test_fused_mx_equals_chained_extreme_scales(empty_groups):
    """MXFP4 with expert scales that put the bf16 gates below, inside, above
    and past the range of the SiLU table (and zero): the fused kernel's
    table lookups and closed forms give the chained kernel's bytes."""
    need_gpu()
    I, K = 128, 256
    # 507 empty groups appended make 513: a launch past the table kernel's
    # 512 groups, which computes the SiLU
    counts = [130, 7, 129, 64, 1, 200] + [0] * empty_groups
    ids = np.array([0, 1, 2, 3, 4, 5] + [g % 6 for g in range(empty_groups)], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    so = Q.padded_scale_offsets(ro)
    rows = int(so[-1])
    a, asf, b, bsf, _ = blockscaled_inputs("mxfp4", int(ro[-1]), 6, 2 * I, K, rows, seed=43)
    es = torch.tensor([1e-36, 1.0, 1e4, 1e38, 0.0, 3e-8], dtype=torch.float32)
    c1, s1, c2, s2 = _fused_and_chained_mx("mxfp4", a, asf, b, bsf, es, ro, so, ids, I, K, rows)
    assert torch.equal(c1, c2)
    assert torch.equal(s1, s2)
    assert moeq.get_device_error() == 0


def test_fused_mx_full_size():
    """128 experts, 16384 tokens top-8 (131072 rows), K = 4096, I = 1536, MXFP4
    throughout: whole buffers equal to the chained path."""
    need_gpu()
    counts = synth.routing_counts(16384, 8, 128, seed=0)
    ro, ids = synth.ragged_groups(counts)
    so = Q.padded_scale_offsets(ro)
    T, I, K, rows = int(ro[-1]), 1536, 4096, int(so[-1])
    a, asf, b, bsf, es = blockscaled_inputs("mxfp4", T, 128, 2 * I, K, rows, seed=90, device=DEV)
    c1, s1, c2, s2 = _fused_and_chained_mx("mxfp4", a, asf, b, bsf, es, ro, so, ids, I, K, rows)
    assert torch.equal(c1, c2)
    assert torch.equal(s1, s2)


def _nvfp4_case(I=192, K=512, seed=21):
    counts = [0, 1, 127, 129, 260, 3]
    ids = np.array([4, 0, 2, 5, 1, 3], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    so = Q.padded_scale_offsets(ro)
    rows = int(so[-1]) + 128
    T = int(ro[-1]) + 5
    a, asf, b, bsf, es = blockscaled_inputs("nvfp4", T, 6, 2 * I, K, rows, seed=seed)
    ots = synth.uniform((6,), 0.05, 0.2, seed=seed + 9)
    return ro, so, ids, rows, T, a, asf, b, bsf, es, ots, I, K


def _fused_nvfp4(case, row_scales):
    ro, so, ids, rows, T, a, asf, b, bsf, es, ots, I, K = case
    c = torch.full((T, I // 2), 0xA5, dtype=torch.uint8, device=DEV)
    s = torch.full((moeq.sf_bytes(rows, I // 16),), 0x5A, dtype=torch.uint8, device=DEV)
    moeq.grouped_matmul_swiglu(c, s, a.to(DEV), asf.to(DEV), b.to(DEV), bsf.to(DEV), es.to(DEV),
                               ots.to(DEV), to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids), I, K,
                               rows, a_row_scales=row_scales)
    torch.cuda.synchronize()
    return c, s


def test_row_scales_of_one_change_nothing():
    need_gpu()
    case = _nvfp4_case()
    T = case[4]
    c0, s0 = _fused_nvfp4(case, None)
    c1, s1 = _fused_nvfp4(case, torch.ones(T, dtype=torch.bfloat16, device=DEV))
    assert torch.equal(c0, c1) and torch.equal(s0, s1)


def test_row_scales_power_of_two_equal_rescaled_chained():
    """With a_row_scales = 2^k per row, gate and up are the chained path's bf16
    y times 2^k exactly, so the fused bytes equal SwiGLU + NVFP4 of that y."""
    need_gpu()
    case = _nvfp4_case(seed=33)
    ro, so, ids, rows, T, a, asf, b, bsf, es, ots, I, K = case
    k = np.random.default_rng(5).integers(-3, 4, T)
    rs = torch.from_numpy(np.ldexp(1.0, k).astype(np.float32)).to(torch.bfloat16)
    c_f, s_f = _fused_nvfp4(case, rs.to(DEV))
    y = torch.zeros((T, 2 * I), dtype=torch.bfloat16, device=DEV)
    moeq.grouped_matmul_blockscaled("nvfp4", y, a.to(DEV), asf.to(DEV), b.to(DEV), bsf.to(DEV),
                                    es.to(DEV), to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids),
                                    2 * I, K, rows)
    y = (y.float() * rs.to(DEV).float()[:, None]).to(torch.bfloat16)   # exact: powers of two
    c_c = torch.full_like(c_f, 0xA5)
    s_c = torch.full_like(s_f, 0x5A)
    moeq.swiglu_quantize(c_c, s_c, y, ots.to(DEV), to_dev_u32(ro), to_dev_u32(so),
                         to_dev_i32(ids), 6, rows)
    torch.cuda.synchronize()
    assert torch.equal(c_f, c_c) and torch.equal(s_f, s_c)


def test_row_scales_against_oracle():
    """General bf16 row scales in [0.5, 2]: the fused output against the
    oracle pipeline (float64 GEMM with expert and row scale, one bf16
    rounding, SwiGLU, NVFP4).  The GPU accumulates in fp32 and rounds
    (acc * s) * r twice, so a gate/up value can differ by one bf16 ulp; the
    bound: at least 99 % of element codes and of block scale codes equal,
    and every scale code within one step."""
    need_gpu()
    case = _nvfp4_case(seed=45)
    ro, so, ids, rows, T, a, asf, b, bsf, es, ots, I, K = case
    rs = synth.uniform((T,), 0.5, 2.0, seed=46).to(torch.bfloat16)
    c_f, s_f = _fused_nvfp4(case, rs.to(DEV))
    y_want = GM.grouped_matmul_blockscaled("nvfp4", a.numpy(), asf.numpy(), b.numpy(), bsf.numpy(),
                                           es.numpy(), ro, so, ids, 2 * I, K, rows,
                                           row_scales=rs.float().numpy())
    yv = F.decode_bf16(y_want)
    want_c, want_s = S.swiglu_quantize(yv, ots.numpy(), ro, so, ids,
                                       out=np.full((T, I // 2), 0xA5, np.uint8),
                                       scales=np.full(L.physical_bytes(rows, I // 16), 0x5A,
                                                      np.uint8), scale_rows_total=rows)
    got_c, got_s = u8(c_f), u8(s_f)
    nrow = int(ro[-1])
    assert np.array_equal(got_c[nrow:], want_c[nrow:])           # rows in no group untouched
    codes_equal = (F.unpack_e2m1(got_c[:nrow]) == F.unpack_e2m1(want_c[:nrow])).mean()
    lg_got, lg_want = L.unswizzle(got_s, rows, I // 16), L.unswizzle(want_s, rows, I // 16)
    assert codes_equal >= 0.99
    assert (lg_got == lg_want).mean() >= 0.99
    assert np.abs(lg_got.astype(int) - lg_want.astype(int)).max() <= 1
