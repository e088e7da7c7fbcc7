"""GPU parity of the grouped quantizer, the per-expert amax -> tensor scale
and the padded scale offsets: bit-exact against the CPU oracle, through the
C ABI, on ragged groups (empty, 1, 127, 128, 129, ... rows), special values,
and the full-size 8-expert / 8192 x 4096 workload on sampled rows."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import moeq, synth
from oracle import formats as F
from oracle import layout as L
from oracle import quantize as Q
from tests._util import DEV, groups_from_counts, need_gpu, sample_rows, to_dev_i32, to_dev_u32, u8

pytestmark = pytest.mark.gpu
FMTS = ["nvfp4", "mxfp8", "mxfp4"]


def _v(fmt):
    return 16 if fmt == "nvfp4" else 32


def _run(fmt, x, ro, so, ids, ts, E, rows, out_fill=0xA5, sf_fill=0x5A):
    T, K = x.shape
    ob = K if fmt == "mxfp8" else K // 2
    out = torch.full((T, ob), out_fill, dtype=torch.uint8, device=DEV)
    sf = torch.full((moeq.sf_bytes(rows, K // _v(fmt)),), sf_fill, dtype=torch.uint8, device=DEV)
    moeq.grouped_quantize(fmt, x, out, sf, to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids),
                          torch.from_numpy(ts).to(DEV) if ts is not None else None, E, rows)
    torch.cuda.synchronize()
    return u8(out), u8(sf)


def _oracle_ts(x_np, ro, ids, E):
    return Q.tensor_scale_from_amax(Q.group_amax(x_np, ro, ids, E))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("K", [128, 384, 1024])
def test_quantize_ragged_small(fmt, K):
    need_gpu()
    counts = [0, 1, 127, 128, 129, 300, 0, 5]
    E = 11
    ids = np.array([3, 7, 0, 10, 2, 5, 9, 1], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    so = Q.padded_scale_offsets(ro)
    T = int(ro[-1]) + 7
    rows = int(so[-1]) + 256
    x = synth.bf16_normal((T, K), 1.0, seed=K, outlier_p=0.01, outlier_scale=50.0)
    x_np = x.float().numpy()
    ts = _oracle_ts(x_np, ro, ids, E)
    out, sf = _run(fmt, x.to(DEV), ro, so, ids, ts, E, rows)
    ob = K if fmt == "mxfp8" else K // 2
    want_out, want_sf = Q.grouped_quantize(
        fmt, x_np, ro, so, ids, ts, out=np.full((T, ob), 0xA5, np.uint8),
        scales=np.full(L.physical_bytes(rows, K // _v(fmt)), 0x5A, np.uint8),
        scale_rows_total=rows)
    assert np.array_equal(out, want_out)
    assert np.array_equal(sf, want_sf)


def _special_rows(K):
    """Rows of bf16 values probing every rounding corner: zeros, -0, bf16
    subnormals, E2M1 / E4M3 midpoints at several scales, huge and tiny
    magnitudes, all-negative blocks."""
    rng = np.random.default_rng(7)
    rows = []
    rows.append(np.zeros(K))
    rows.append(-np.zeros(K))
    rows.append(np.full(K, 2.0 ** -133))                     # smallest bf16 subnormal
    rows.append(rng.choice([-1, 1], K) * 2.0 ** rng.integers(-133, -120, K))
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 7.0, 0.1])
    rows.append(np.resize(np.concatenate([[6.0], mids]), K))
    rows.append(np.resize(np.concatenate([[448.0], mids * 64]), K))
    rows.append(-np.abs(rng.normal(0, 1, K)))
    rows.append(rng.normal(0, 1, K) * 1e30)
    rows.append(rng.normal(0, 1, K) * 1e-30)
    r = rng.normal(0, 1, K)
    r[::16] = 0.0
    r[1::33] = -0.0
    rows.append(r)
    for s in (1e-3, 1.0, 3e3):
        rows.append(rng.normal(0, s, K))
    x = np.stack(rows)
    return F.round_bf16(x).astype(np.float32)


@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_special_values(fmt):
    need_gpu()
    K = 256
    xs = _special_rows(K)
    n = xs.shape[0]
    # one group per row, each its own expert, with very different tensor scales
    ro, ids = groups_from_counts([1] * n)
    so = Q.padded_scale_offsets(ro)
    ts = np.geomspace(1e-6, 1e3, n).astype(np.float32)
    rows = int(so[-1])
    x = torch.from_numpy(xs).to(torch.bfloat16)
    out, sf = _run(fmt, x.to(DEV), ro, so, ids, ts, n, rows)
    want_out, want_sf = Q.grouped_quantize(fmt, xs, ro, so, ids, ts, out=np.full_like(out, 0xA5),
                                           scales=np.full_like(sf, 0x5A), scale_rows_total=rows)
    assert np.array_equal(out, want_out)
    assert np.array_equal(sf, want_sf)


@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_strided_rows(fmt):
    """Rows 16- but not 32-byte aligned (row stride K + 8 elements, and a
    view starting 8 elements in): the kernel's two-16-byte-load path."""
    need_gpu()
    counts = [3, 130, 0, 40]
    ro, ids = groups_from_counts(counts, [1, 0, 3, 2])
    so = Q.padded_scale_offsets(ro)
    T, K, E = int(ro[-1]), 256, 4
    rows = int(so[-1])
    base = synth.bf16_normal((T, K + 16), 1.0, seed=8)
    view = base[:, 8:8 + K]
    x_np = view.float().numpy()
    ts = _oracle_ts(x_np, ro, ids, E)
    dev_base = base.to(DEV)
    x_dev = dev_base[:, 8:8 + K]
    assert x_dev.stride(0) == K + 16 and (x_dev.data_ptr() % 32) != 0
    ob = K if fmt == "mxfp8" else K // 2
    out = torch.full((T, ob), 0xA5, dtype=torch.uint8, device=DEV)
    sf = torch.full((moeq.sf_bytes(rows, K // _v(fmt)),), 0x5A, dtype=torch.uint8, device=DEV)
    moeq.grouped_quantize(fmt, x_dev, out, sf, to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids),
                          torch.from_numpy(ts).to(DEV), E, rows)
    want_out, want_sf = Q.grouped_quantize(fmt, x_np, ro, so, ids, ts,
                                           out=np.full((T, ob), 0xA5, np.uint8),
                                           scales=np.full(L.physical_bytes(rows, K // _v(fmt)), 0x5A,
                                                          np.uint8), scale_rows_total=rows)
    assert np.array_equal(u8(out), want_out) and np.array_equal(u8(sf), want_sf)
    amax = torch.empty(E, device=DEV)
    moeq.grouped_amax_scale(x_dev, to_dev_u32(ro), to_dev_i32(ids), amax, E)
    assert np.array_equal(amax.cpu().numpy().view(np.uint32), ts.view(np.uint32))


def _cfg2(seed=0):
    counts = synth.routing_counts(4096, 2, 8, seed=seed)
    ro, ids = synth.ragged_groups(counts)
    x = synth.bf16_normal((int(ro[-1]), 4096), 1.0, seed=seed, device=DEV, outlier_p=0.001,
                          outlier_scale=50.0)
    return ro, ids, x


@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_full_size_sampled(fmt):
    """8 experts, 4096 tokens top-2 -> 8192 rows, hidden 4096 (the grouped
    activation-quantize workload), checked on sampled rows and on every
    padding row."""
    need_gpu()
    ro, ids, x = _cfg2()
    E, K = 8, 4096
    so = Q.padded_scale_offsets(ro)
    rows = int(so[-1])
    x_np = x.float().cpu().numpy()
    ts = _oracle_ts(x_np, ro, ids, E)
    out, sf = _run(fmt, x, ro, so, ids, ts, E, rows)
    kv = K // _v(fmt)
    lg = L.unswizzle(sf, rows, kv)
    sel = sample_rows(ro, 256, seed=1)
    for g in range(len(ids)):
        r0, r1 = int(ro[g]), int(ro[g + 1])
        pick = sel[(sel >= r0) & (sel < r1)]
        q, sc = Q.quantize_rows(fmt, x_np[pick], ts[ids[g]] if fmt == "nvfp4" else None)
        assert np.array_equal(out[pick], q)
        assert np.array_equal(lg[int(so[g]) + pick - r0], sc)
        assert not lg[int(so[g]) + r1 - r0:int(so[g + 1])].any()


def test_amax_scale_bit_exact():
    need_gpu()
    counts = [0, 3, 129, 1, 700]
    ids = np.array([4, 2, 0, 2, 5], np.int32)            # expert 2 twice, 1 and 3 unused
    ro, ids = groups_from_counts(counts, ids)
    E, K = 6, 512
    T = int(ro[-1]) + 5
    x = synth.bf16_normal((T, K), 1.0, seed=3, outlier_p=0.002, outlier_scale=1e4)
    x[-5:] = 1e6                                          # rows in no group are ignored
    out = torch.full((E,), -1.0, device=DEV)
    moeq.grouped_amax_scale(x.to(DEV), to_dev_u32(ro), to_dev_i32(ids), out, E)
    got = out.cpu().numpy()
    want = _oracle_ts(x.float().numpy(), ro, ids, E)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_amax_scale_full_size():
    need_gpu()
    ro, ids, x = _cfg2(seed=2)
    out = torch.empty(8, device=DEV)
    moeq.grouped_amax_scale(x, to_dev_u32(ro), to_dev_i32(ids), out, 8)
    want = _oracle_ts(x.float().cpu().numpy(), ro, ids, 8)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("T", [65535, 65539])
def test_amax_scale_launch_shapes(T):
    """Both launch shapes of the amax pass: below 65536 rows one row per warp
    in 4-warp CTAs (65535: the last CTA has 3 warps), from 65536 rows two
    rows per warp in 8-warp CTAs (65539: the last warp has one row); the
    largest value of each expert lies in its group's last rows."""
    need_gpu()
    K, E = 128, 5
    counts = [T // 4, 0, T // 4, T - 3 * (T // 4) - 7, T // 4 + 7]
    ids = np.array([3, 1, 0, 4, 2], np.int32)
    ro, ids = groups_from_counts(counts, ids)
    assert int(ro[-1]) == T
    x = synth.bf16_normal((T, K), 1.0, seed=5)
    for g in range(len(counts)):
        if counts[g]:
            x[int(ro[g + 1]) - 1, (17 * g) % K] = -300.0 - g   # tail row of the group
    out = torch.full((E,), -1.0, device=DEV)
    moeq.grouped_amax_scale(x.to(DEV), to_dev_u32(ro), to_dev_i32(ids), out, E)
    want = _oracle_ts(x.float().numpy(), ro, ids, E)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32))
    # expert 1 has no rows (scale 1); expert 3's amax is its group's tail value 300
    assert want[1] == 1.0 and want[3] == np.float32(300.0) / np.float32(2688.0)


def test_padded_scale_offsets():
    need_gpu()
    rng = np.random.default_rng(4)
    for G in (1, 7, 33, 256, 1000):
        counts = rng.integers(0, 300, G)
        counts[rng.random(G) < 0.2] = 0
        ro, _ = groups_from_counts(counts)
        so = torch.full((G + 1,), -1, dtype=torch.int32, device=DEV)
        moeq.padded_scale_offsets(to_dev_u32(ro), so)
        got = so.cpu().numpy().view(np.uint32)
        assert np.array_equal(got, Q.padded_scale_offsets(ro))


def test_quantize_no_groups_is_noop():
    need_gpu()
    x = torch.zeros((4, 128), dtype=torch.bfloat16, device=DEV)
    out = torch.full((4, 64), 7, dtype=torch.uint8, device=DEV)
    sf = torch.full((512,), 9, dtype=torch.uint8, device=DEV)
    e = torch.zeros(0, dtype=torch.int32, device=DEV)
    o = torch.zeros(1, dtype=torch.int32, device=DEV)
    moeq.grouped_quantize("nvfp4", x, out, sf, o, o, e, torch.ones(1, device=DEV), 1, 128,
                          num_active_experts=0)
    torch.cuda.synchronize()
    assert (out == 7).all() and (sf == 9).all()


def test_quantize_bad_device_data_sets_error_and_skips_group():
    need_gpu()
    moeq.clear_device_error()
    counts = [10, 20, 30]
    ro, _ = groups_from_counts(counts)
    ids = np.array([0, 9, 1], np.int32)                  # 9 is out of range (E = 2)
    so = Q.padded_scale_offsets(ro)
    K = 128
    x = synth.bf16_normal((60, K), 1.0, seed=5)
    ts = np.ones(2, np.float32)
    out, sf = _run("nvfp4", x.to(DEV), ro, so, ids, ts, 2, int(so[-1]))
    bits = moeq.get_device_error()
    assert bits & moeq.DEVERR_BAD_EXPERT
    assert np.all(out[10:30] == 0xA5)                    # the bad group is skipped
    good_ids = ids.copy()
    good_ids[1] = 0
    want_out, _ = Q.grouped_quantize("nvfp4", x.float().numpy(), ro, so, good_ids, ts,
                                     out=np.full_like(out, 0xA5), scale_rows_total=int(so[-1]))
    assert np.array_equal(out[:10], want_out[:10]) and np.array_equal(out[30:], want_out[30:])
    # non-monotone offsets: flagged, nothing faults, the GPU stays usable
    moeq.clear_device_error()
    bad_ro = np.array([0, 40, 20, 60], np.uint32)
    _run("mxfp8", x.to(DEV), bad_ro, np.array([0, 128, 256, 384], np.uint32), np.array([0, 1, 1]),
         None, 2, 384)
    assert moeq.get_device_error() & (moeq.DEVERR_BAD_OFFSETS | moeq.DEVERR_SCALE_ROWS)
    moeq.clear_device_error()
    assert moeq.get_device_error() == 0


@pytest.mark.parametrize("fmt", FMTS)
def test_quantize_gather_bit_exact(fmt):
    """Gather-fused quantize: quantized row t reads input row indices[t] / top_k
    (expert-sorted routing positions), bit-exact against the oracle on the
    gathered rows; also the gathered per-expert amax."""
    need_gpu()
    tokens, top_k, E, K = 300, 3, 8, 512
    rng = np.random.default_rng(31)
    experts = np.stack([rng.choice(E, top_k, replace=False) for _ in range(tokens)])
    pos = np.arange(tokens * top_k)
    order = np.argsort(experts.reshape(-1), kind="stable")
    indices = pos[order].astype(np.int32)
    counts = np.bincount(experts.reshape(-1), minlength=E)
    ro, ids = synth.ragged_groups(counts)
    so = Q.padded_scale_offsets(ro)
    rows = int(so[-1])
    x = synth.bf16_normal((tokens, K), 1.0, seed=9, outlier_p=0.01, outlier_scale=30.0)
    xg = Q.gather_rows(x.float().numpy(), indices, top_k)
    ts = _oracle_ts(xg, ro, ids, E)
    T = len(indices)
    idx_d = torch.from_numpy(indices).to(DEV)
    amax = torch.empty(E, device=DEV)
    moeq.grouped_amax_scale_gather(x.to(DEV), idx_d, top_k, to_dev_u32(ro), to_dev_i32(ids), amax, E)
    assert np.array_equal(amax.cpu().numpy().view(np.uint32), ts.view(np.uint32))
    ob = K if fmt == "mxfp8" else K // 2
    out = torch.full((T, ob), 0xA5, dtype=torch.uint8, device=DEV)
    sf = torch.full((moeq.sf_bytes(rows, K // _v(fmt)),), 0x5A, dtype=torch.uint8, device=DEV)
    moeq.grouped_quantize_gather(fmt, x.to(DEV), idx_d, top_k, out, sf, to_dev_u32(ro),
                                 to_dev_u32(so), to_dev_i32(ids), amax, E, rows)
    want_out, want_sf = Q.grouped_quantize(fmt, xg, ro, so, ids, ts,
                                           out=np.full((T, ob), 0xA5, np.uint8),
                                           scales=np.full(L.physical_bytes(rows, K // _v(fmt)), 0x5A,
                                                          np.uint8), scale_rows_total=rows)
    assert np.array_equal(u8(out), want_out) and np.array_equal(u8(sf), want_sf)


def test_quantize_gather_bad_index_flagged():
    need_gpu()
    moeq.clear_device_error()
    K, E = 128, 2
    ro, ids = groups_from_counts([3, 2])
    so = Q.padded_scale_offsets(ro)
    x = synth.bf16_normal((4, K), 1.0, seed=10)
    indices = torch.tensor([0, 1, 9, 2, 3], dtype=torch.int32, device=DEV)   # 9 -> row 9 > 3
    out = torch.full((5, K // 2), 0xA5, dtype=torch.uint8, device=DEV)
    sf = torch.zeros(moeq.sf_bytes(int(so[-1]), K // 16), dtype=torch.uint8, device=DEV)
    moeq.grouped_quantize_gather("nvfp4", x.to(DEV), indices, 1, out, sf, to_dev_u32(ro),
                                 to_dev_u32(so), to_dev_i32(ids), torch.ones(E, device=DEV), E,
                                 int(so[-1]))
    assert moeq.get_device_error() & moeq.DEVERR_BAD_INDEX
    assert (out[2] == 0xA5).all() and not (out[0] == 0xA5).all()
    moeq.clear_device_error()
