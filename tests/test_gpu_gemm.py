"""GPU parity of the grouped GEMMs through the C ABI: the rowwise FP8 GEMM and
the NVFP4 / MXFP8 block-scaled GEMM against the float64 CPU oracle (per
element within max(2 bf16 ulp, 1e-3 rms)), on ragged multi-tile cases with
empty groups and permuted expert ids, the tiny 3-group case, the MoE-scale
and decode-shaped workloads on sampled rows, and exact GPU-vs-GPU
invariants (power-of-two scaling, group permutation, canaries)."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import moeq, synth
from oracle import gemm as OG
from oracle import layout as L
from tests._util import (DEV, assert_gemm_close, bf16_bits, group_sample_rows,
                         groups_from_counts, need_gpu, sample_rows, tile_sample_cols, to_dev_i32,
                         to_dev_u32, u8)

pytestmark = pytest.mark.gpu
CANARY = -12288.0   # exactly representable in bf16


# ----------------------------------------------------------- FP8 rowwise

def _rowwise_inputs(T, E, N, K, seed, a_std=1.0, b_std=0.5, device="cpu"):
    a = synth.e4m3_normal((T, K), a_std, seed=seed, device=device)
    b = synth.e4m3_normal((E, N, K), b_std, seed=seed + 1, device=device)
    sa = synth.uniform((T,), 0.01, 0.1, seed=seed + 2, device=device)
    sb = synth.uniform((E, N), 0.005, 0.05, seed=seed + 3, device=device)
    return a, b, sa, sb


def _assert_all_written(c):
    """Every row of these outputs lies in a group: no element may keep the
    canary the buffer was filled with (their outputs are far from -12288)."""
    assert not bool(torch.any(c == CANARY))


def _run_rowwise(a, b, sa, sb, ro, ids, T=None):
    T = a.shape[0] if T is None else T
    c = torch.full((T, b.shape[1]), CANARY, dtype=torch.bfloat16, device=DEV)
    moeq.grouped_matmul_rowwise_fp8(c, a.to(DEV), b.to(DEV), sa.to(DEV), sb.to(DEV),
                                    to_dev_u32(ro), to_dev_i32(ids))
    torch.cuda.synchronize()
    return c


def _check_rowwise(c, a, b, sa, sb, ro, ids):
    out = bf16_bits(c)
    _, f64 = OG.grouped_matmul_rowwise_fp8(u8(a), u8(b), sa.numpy(), sb.numpy(), ro, ids,
                                           return_f64=True)
    T = out.shape[0]
    written = np.zeros(T, bool)
    written[int(ro[0]):int(ro[-1])] = True
    assert_gemm_close(out, f64, mask_rows=written)
    canary = np.float32(CANARY).view(np.uint32) >> 16
    assert np.all(out[~written] == canary)


def test_rowwise_fp8_tiny_three_groups():
    """E = 4, groups [7, 16, 9] rows on experts [2, 0, 3], K = 128, N = 64."""
    need_gpu()
    ro = np.array([0, 7, 23, 32], np.uint32)
    ids = np.array([2, 0, 3], np.int32)
    a, b, sa, sb = _rowwise_inputs(32, 4, 64, 128, seed=0)
    c = _run_rowwise(a, b, sa, sb, ro, ids)
    _check_rowwise(c, a, b, sa, sb, ro, ids)


@pytest.mark.parametrize("N,K", [(512, 512), (80, 256), (64, 1024), (272, 128)])
def test_rowwise_fp8_ragged_multitile(N, K):
    need_gpu()
    counts = [0, 1, 127, 128, 129, 300, 0, 2]
    ids = np.array([5, 0, 3, 1, 7, 2, 4, 6], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    T = int(ro[-1]) + 9                                  # trailing rows in no group
    a, b, sa, sb = _rowwise_inputs(T, 8, N, K, seed=N + K)
    c = _run_rowwise(a, b, sa, sb, ro, ids)
    _check_rowwise(c, a, b, sa, sb, ro, ids)


def test_rowwise_fp8_exact_invariants():
    need_gpu()
    counts = [130, 0, 257, 64]
    ro, ids = groups_from_counts(counts, [2, 1, 0, 3])
    T = int(ro[-1])
    a, b, sa, sb = _rowwise_inputs(T, 4, 256, 512, seed=9)
    c1 = bf16_bits(_run_rowwise(a, b, sa, sb, ro, ids))
    # doubling every a_scale doubles every output exactly
    c2 = bf16_bits(_run_rowwise(a, b, sa * 2, sb, ro, ids))
    v1 = (c1.astype(np.uint32) << 16).view(np.float32)
    v2 = (c2.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(v1 * 2, v2)
    # permuting the groups (rows and expert ids together) permutes the rows
    perm = [2, 3, 0, 1]
    rows = [np.arange(ro[g], ro[g + 1]) for g in range(4)]
    idx = np.concatenate([rows[g] for g in perm]).astype(np.int64)
    ro_p, ids_p = groups_from_counts([counts[g] for g in perm], ids[perm])
    ti = torch.from_numpy(idx)
    a_p = a.view(torch.uint8)[ti].view(torch.float8_e4m3fn)
    cp = bf16_bits(_run_rowwise(a_p, b, sa[ti], sb, ro_p, ids_p))
    assert np.array_equal(cp, c1[idx])


def _full_width_groups(ro):
    """Groups checked over every output column: the first, the largest, the
    smallest non-empty and the last."""
    n = np.diff(ro.astype(np.int64))
    nz = np.nonzero(n)[0]
    return sorted({int(nz[0]), int(np.argmax(n)), int(nz[np.argmin(n[nz])]), int(nz[-1])})


def _all_rows(ro):
    return [np.arange(int(ro[g]), int(ro[g + 1]), dtype=np.int64) for g in range(len(ro) - 1)]


def _rows_cols(t, rows, cols=None):
    """uint8 numpy copy of t[rows] (and [:, cols]), gathered on the device."""
    if t.dtype != torch.uint8:
        t = t.view(torch.uint8)
    idx = torch.from_numpy(np.asarray(rows, np.int64)).to(t.device)
    sub = t.index_select(0, idx)
    if cols is not None:
        sub = sub.index_select(1, torch.from_numpy(np.asarray(cols, np.int64)).to(t.device))
    return u8(sub)


def _check_rowwise_sampled(c, a, sa, b, sb, ro, ids, N, tile, all_rows=False):
    """Every non-empty group: rows of its first, middle and last m-block (or
    all its rows) against the oracle, on columns spread over every n-tile
    (all columns for a few groups).  Tensors on the device: c [T, N] bf16,
    a [T, K] e4m3, sa [T], b [E, N, K] e4m3, sb [E, N]."""
    cols = tile_sample_cols(N, tile)
    full = _full_width_groups(ro)
    checked = 0
    sa_np = sa.cpu().numpy()
    for g, rows in enumerate(_all_rows(ro) if all_rows else group_sample_rows(ro)):
        if rows.size == 0:
            continue
        e = int(ids[g])
        cc = np.arange(N) if g in full else cols
        _, f64 = OG.grouped_matmul_rowwise_fp8(_rows_cols(a, rows), _rows_cols(b[e], cc)[None],
                                               sa_np[rows], sb[e:e + 1, torch.from_numpy(cc).to(
                                                   sb.device)].cpu().numpy(),
                                               np.array([0, len(rows)], np.uint32), [0],
                                               return_f64=True)
        got = bf16_bits(c.index_select(0, torch.from_numpy(rows).to(c.device)))[:, cc]
        assert_gemm_close(got, f64)
        checked += 1
    assert checked == int((np.diff(ro.astype(np.int64)) > 0).sum())


def test_rowwise_fp8_moe_scale_sampled():
    """64 experts, 8192 tokens top-8 with Zipf(1.1) popularity -> 65536 rows,
    K = 7168, N = 4096: every group on rows of its first, middle and last
    m-block."""
    need_gpu()
    counts = synth.routing_counts(8192, 8, 64, seed=0, zipf_s=1.1)
    ro, ids = synth.ragged_groups(counts)
    T, E, N, K = int(ro[-1]), 64, 4096, 7168
    a, sa = synth.fp8_rowwise((T, K), 1.0, seed=10, device=DEV)
    b, sb = synth.fp8_rowwise((E, N, K), 0.02, seed=11, device=DEV)
    c = torch.full((T, N), CANARY, dtype=torch.bfloat16, device=DEV)
    moeq.grouped_matmul_rowwise_fp8(c, a, b, sa, sb.reshape(E, N), to_dev_u32(ro),
                                    to_dev_i32(ids), max_tokens_per_expert=int(counts.max()))
    torch.cuda.synchronize()
    _assert_all_written(c)
    _check_rowwise_sampled(c, a, sa, b, sb.reshape(E, N), ro, ids, N, 256)


def test_rowwise_fp8_decode_shape_sampled():
    """256 experts, 64 tokens top-8 -> 512 rows over ~224 experts of 1-7 rows:
    every group, all its rows."""
    need_gpu()
    counts = synth.routing_counts(64, 8, 256, seed=0)
    ro, ids = synth.ragged_groups(counts)
    T, E, N, K = int(ro[-1]), 256, 4096, 7168
    a, sa = synth.fp8_rowwise((T, K), 1.0, seed=20, device=DEV)
    b, sb = synth.fp8_rowwise((E, N, K), 0.02, seed=21, device=DEV)
    c = torch.full((T, N), CANARY, dtype=torch.bfloat16, device=DEV)
    moeq.grouped_matmul_rowwise_fp8(c, a, b, sa, sb.reshape(E, N), to_dev_u32(ro),
                                    to_dev_i32(ids), max_tokens_per_expert=int(counts.max()))
    torch.cuda.synchronize()
    _assert_all_written(c)
    _check_rowwise_sampled(c, a, sa, b, sb.reshape(E, N), ro, ids, N, 256, all_rows=True)


def test_rowwise_fp8_bad_expert_skips_group():
    need_gpu()
    moeq.clear_device_error()
    ro, _ = groups_from_counts([50, 60, 70])
    ids = np.array([1, -3, 0], np.int32)
    a, b, sa, sb = _rowwise_inputs(180, 2, 128, 128, seed=30)
    c = bf16_bits(_run_rowwise(a, b, sa, sb, ro, ids))
    assert moeq.get_device_error() & moeq.DEVERR_BAD_EXPERT
    canary = np.float32(CANARY).view(np.uint32) >> 16
    assert np.all(c[50:110] == canary)
    good = np.array([1, 0, 0], np.int32)
    _, f64 = OG.grouped_matmul_rowwise_fp8(u8(a), u8(b), sa.numpy(), sb.numpy(), ro, good,
                                           return_f64=True)
    keep = np.r_[0:50, 110:180]
    assert_gemm_close(c[keep], f64[keep])
    moeq.clear_device_error()


# --------------------------------------------------------- block-scaled

def blockscaled_inputs(fmt, T, E, N, K, rows, seed, device="cpu", a_sf=(0x20, 0x30),
                       b_sf=(0x18, 0x28)):
    """Random quantized operands: elements, tiled scale buffers (random
    codes everywhere), expert scales."""
    if fmt == "nvfp4":
        a = synth.random_fp4_packed((T, K // 2), seed=seed, device=device)
        b = synth.random_fp4_packed((E, N, K // 2), seed=seed + 1, device=device)
        kv = K // 16
        lo_a, hi_a = a_sf
        lo_b, hi_b = b_sf
    elif fmt == "mxfp4":
        a = synth.random_fp4_packed((T, K // 2), seed=seed, device=device)
        b = synth.random_fp4_packed((E, N, K // 2), seed=seed + 1, device=device)
        kv = K // 32
        lo_a, hi_a, lo_b, hi_b = 118, 130, 116, 126
    else:
        a = synth.e4m3_normal((T, K), 1.0, seed=seed, device=device).view(torch.uint8)
        b = synth.e4m3_normal((E, N, K), 1.0, seed=seed + 1, device=device).view(torch.uint8)
        kv = K // 32
        lo_a, hi_a, lo_b, hi_b = 118, 130, 116, 126
    asf = synth.random_bytes(moeq.sf_bytes(rows, kv), lo_a, hi_a, seed=seed + 2, device=device)
    bsf = synth.random_bytes(E * moeq.sf_bytes(N, kv), lo_b, hi_b, seed=seed + 3, device=device)
    es = synth.uniform((E,), 0.5, 2.0, seed=seed + 4, device=device)
    return a, asf, b, bsf, es


def run_blockscaled(fmt, a, asf, b, bsf, es, ro, so, ids, N, K, rows):
    T = a.shape[0]
    c = torch.full((T, N), CANARY, dtype=torch.bfloat16, device=DEV)
    moeq.grouped_matmul_blockscaled(fmt, c, a.to(DEV), asf.to(DEV), b.to(DEV), bsf.to(DEV),
                                    None if es is None else es.to(DEV), to_dev_u32(ro),
                                    to_dev_u32(so), to_dev_i32(ids), N, K, rows)
    torch.cuda.synchronize()
    return c


@pytest.mark.parametrize("fmt,es_on", [("nvfp4", True), ("mxfp8", False), ("mxfp8", True),
                                       ("mxfp4", False), ("mxfp4", True)])
# N = 384 and 1152: with the FP4 kinds' 256-column tiles the last n-tile lies
# half past N
@pytest.mark.parametrize("N,K", [(256, 512), (128, 1024), (512, 1536), (384, 512), (1152, 256)])
def test_blockscaled_ragged_multitile(fmt, es_on, N, K):
    need_gpu()
    from oracle import quantize as Q
    counts = [0, 1, 127, 129, 260, 3]
    ids = np.array([4, 0, 2, 5, 1, 3], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    so = Q.padded_scale_offsets(ro)
    rows = int(so[-1]) + 128
    T = int(ro[-1]) + 5
    a, asf, b, bsf, es = blockscaled_inputs(fmt, T, 6, N, K, rows, seed=N + K)
    es = es if es_on else None
    c = bf16_bits(run_blockscaled(fmt, a, asf, b, bsf, es, ro, so, ids, N, K, rows))
    _, f64 = OG.grouped_matmul_blockscaled(fmt, u8(a), u8(asf), u8(b), u8(bsf),
                                           None if es is None else es.numpy(), ro, so, ids,
                                           N=N, K=K, scale_rows_total=rows, return_f64=True)
    written = np.zeros(T, bool)
    written[:int(ro[-1])] = True
    assert_gemm_close(c, f64, mask_rows=written)
    canary = np.float32(CANARY).view(np.uint32) >> 16
    assert np.all(c[~written] == canary)


def _cfg4_groups(seed=0):
    from oracle import quantize as Q
    counts = synth.routing_counts(16384, 8, 128, seed=seed)
    ro, ids = synth.ragged_groups(counts)
    so = Q.padded_scale_offsets(ro)
    return counts, ro, ids, so


def _check_blockscaled_sampled(fmt, c, a, asf_np, b, bsf_np, es_np, ro, so, ids, N, K,
                               tile, all_rows=False):
    """Every non-empty group: rows of its first, middle and last m-block (or
    all its rows) against the oracle, each as a one-group problem over its
    own scale rows and the sampled weight rows (columns) with theirs.  c, a,
    b on the device; the scale buffers as numpy bytes."""
    v = 16 if fmt == "nvfp4" else 32
    kv = K // v
    per = moeq.sf_bytes(N, kv)
    cols = tile_sample_cols(N, tile)
    full = _full_width_groups(ro)
    kcols = np.arange(kv)[None, :]
    checked = 0
    for g, rows in enumerate(_all_rows(ro) if all_rows else group_sample_rows(ro)):
        if rows.size == 0:
            continue
        e = int(ids[g])
        cc = np.arange(N) if g in full else cols
        prow = int(so[g]) + rows - int(ro[g])
        pad = np.zeros((128, kv), np.uint8)
        pad[:len(rows)] = asf_np[L.sf_offset(prow[:, None], kcols, kv)]
        bsf_e = bsf_np[e * per:(e + 1) * per]
        sub_bsf = L.swizzle(bsf_e[L.sf_offset(cc[:, None], kcols, kv)])
        _, f64 = OG.grouped_matmul_blockscaled(
            fmt, _rows_cols(a, rows), L.swizzle(pad), _rows_cols(b[e], cc)[None], sub_bsf,
            None if es_np is None else es_np[e:e + 1], np.array([0, len(rows)], np.uint32),
            np.array([0, 128], np.uint32), [0], N=len(cc), K=K, scale_rows_total=128,
            return_f64=True)
        got = bf16_bits(c.index_select(0, torch.from_numpy(rows).to(c.device)))[:, cc]
        assert_gemm_close(got, f64)
        checked += 1
    assert checked == int((np.diff(ro.astype(np.int64)) > 0).sum())


def test_nvfp4_blockscaled_moe_scale_sampled():
    """128 experts, 16384 tokens top-8 -> 131072 rows, K = 4096, N = 3072:
    every group on rows of its first, middle and last m-block."""
    need_gpu()
    counts, ro, ids, so = _cfg4_groups()
    T, E, N, K = int(ro[-1]), 128, 3072, 4096
    rows = int(so[-1])
    a, asf, b, bsf, es = blockscaled_inputs("nvfp4", T, E, N, K, rows, seed=40, device=DEV)
    c = run_blockscaled("nvfp4", a, asf, b, bsf, es, ro, so, ids, N, K, rows)
    _assert_all_written(c)
    _check_blockscaled_sampled("nvfp4", c, a, u8(asf), b, u8(bsf), es.cpu().numpy(),
                               ro, so, ids, N, K, 256)


def test_nvfp4_down_projection_shape_sampled():
    """The MoE layer's down-projection: 128 experts, 16384 tokens top-8 ->
    131072 rows, K = 1536, N = 4096 (a short mainloop, so the bf16 epilogue's
    staged tensor stores and the lanes' masked stores of chunks that reach
    past a group's end carry most of the output): every group on rows of its
    first, middle and last m-block."""
    need_gpu()
    counts, ro, ids, so = _cfg4_groups(seed=2)
    T, E, N, K = int(ro[-1]), 128, 4096, 1536
    rows = int(so[-1])
    a, asf, b, bsf, es = blockscaled_inputs("nvfp4", T, E, N, K, rows, seed=60, device=DEV)
    c = run_blockscaled("nvfp4", a, asf, b, bsf, es, ro, so, ids, N, K, rows)
    _assert_all_written(c)
    _check_blockscaled_sampled("nvfp4", c, a, u8(asf), b, u8(bsf), es.cpu().numpy(),
                               ro, so, ids, N, K, 256)


def test_mxfp8_decode_shape_sampled():
    """256 experts, 64 tokens top-8 -> 512 rows, K = 7168, N = 4096, MXFP8:
    every group, all its rows."""
    need_gpu()
    from oracle import quantize as Q
    counts = synth.routing_counts(64, 8, 256, seed=0)
    ro, ids = synth.ragged_groups(counts)
    so = Q.padded_scale_offsets(ro)
    T, E, N, K = int(ro[-1]), 256, 4096, 7168
    rows = int(so[-1])
    a, asf, b, bsf, _ = blockscaled_inputs("mxfp8", T, E, N, K, rows, seed=50, device=DEV)
    c = run_blockscaled("mxfp8", a, asf, b, bsf, None, ro, so, ids, N, K, rows)
    _assert_all_written(c)
    _check_blockscaled_sampled("mxfp8", c, a, u8(asf), b, u8(bsf), None, ro, so, ids,
                               N, K, 128, all_rows=True)


def test_mxfp4_blockscaled_moe_scale_sampled():
    """MXFP4 at the 128-expert shape (K = 4096, N = 3072): every group on rows
    of its first, middle and last m-block."""
    need_gpu()
    counts, ro, ids, so = _cfg4_groups(seed=1)
    T, E, N, K = int(ro[-1]), 128, 3072, 4096
    rows = int(so[-1])
    a, asf, b, bsf, _ = blockscaled_inputs("mxfp4", T, E, N, K, rows, seed=45, device=DEV)
    c = run_blockscaled("mxfp4", a, asf, b, bsf, None, ro, so, ids, N, K, rows)
    _assert_all_written(c)
    _check_blockscaled_sampled("mxfp4", c, a, u8(asf), b, u8(bsf), None, ro, so, ids,
                               N, K, 256)


