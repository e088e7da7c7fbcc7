"""Single-rank expert dispatch on the GPU ("Struct_ep_dispatch_mxfp4",
execute; the exchange is the identity with one rank) against the oracle:
the routing is integer work and must match exactly (row offsets, expert
ids, source choices, scale offsets); the MXFP4 rows and their E8M0 scales
must match byte for byte, in the padded and in the fixed-slot scale layout;
the slot layout must feed the MXFP4 GEMM to the same result."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import moeq, synth
from oracle import dispatch as D
from oracle import layout as L
from oracle import quantize as Q
from tests._util import DEV, need_gpu, note, u8

pytestmark = pytest.mark.gpu


def _topk(T, k, E, seed, zipf=None):
    rng = np.random.default_rng(seed)
    p = None
    if zipf:
        p = (np.arange(1, E + 1) ** -zipf)
        p = p / p.sum()
    return np.stack([rng.choice(E, k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def _route_gpu(ids, E, slot_rows=0):
    n = ids.size
    ro = torch.full((E + 1,), -1, dtype=torch.int32, device=DEV)
    eids = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    src = torch.full((max(n, 1),), -7, dtype=torch.int32, device=DEV)
    so = torch.full((E + 1,), -1, dtype=torch.int32, device=DEV)
    moeq.route_topk(torch.from_numpy(ids).to(DEV), ro, eids, src, so, slot_rows)
    torch.cuda.synchronize()
    return (ro.cpu().numpy().view(np.uint32), eids.cpu().numpy(), src.cpu().numpy(),
            so.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("T,k,E,zipf", [(3, 2, 3, None), (129, 2, 8, None), (64, 8, 256, None),
                                        (1000, 4, 33, 1.1), (16384, 8, 128, None),
                                        (5000, 6, 1024, None)])
def test_route_matches_oracle(T, k, E, zipf):
    need_gpu()
    moeq.clear_device_error()
    ids = (np.array([[2, 0], [1, 2], [0, 0]], np.int32) if T == 3
           else _topk(T, k, E, seed=T + E, zipf=zipf))
    ro, eids, src, dropped = D.route_topk(ids, E)
    g_ro, g_eids, g_src, g_so = _route_gpu(ids, E)
    assert dropped == 0
    assert np.array_equal(g_ro, ro)
    assert np.array_equal(g_eids, eids)
    assert np.array_equal(g_src[:len(src)], src)
    assert np.array_equal(g_so, Q.padded_scale_offsets(ro))
    _, _, _, g_slot = _route_gpu(ids, E, slot_rows=256)
    assert np.array_equal(g_slot, D.slot_scale_offsets(E, 256))
    assert moeq.get_device_error() == 0
    note(choices=int(ids.size), experts=E)


def test_route_drops_invalid_ids():
    need_gpu()
    moeq.clear_device_error()
    ids = _topk(200, 3, 10, seed=1)
    ids[5, 1] = -1
    ids[77, 0] = 10
    ids[199, 2] = 1 << 30
    ro, _, src, dropped = D.route_topk(ids, 10)
    g_ro, _, g_src, _ = _route_gpu(ids, 10)
    assert dropped == 3
    assert np.array_equal(g_ro, ro)
    assert np.array_equal(g_src[:len(src)], src)
    assert np.all(g_src[len(src):] == -7)          # entries past the routed rows untouched
    assert moeq.get_device_error() & moeq.DEVERR_BAD_EXPERT
    moeq.clear_device_error()


def _dispatch_gpu(tok, ids, E, slot_rows=0):
    T, H = tok.shape
    k = ids.shape[1]
    rows = moeq.dispatch_scale_rows(T, k, E, slot_rows)
    out = torch.full((T * k, H // 2), 0xA5, dtype=torch.uint8, device=DEV)
    sf = torch.full((moeq.sf_bytes(rows, H // 32),), 0x5A, dtype=torch.uint8, device=DEV)
    ro = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    eids = torch.empty(E, dtype=torch.int32, device=DEV)
    src = torch.empty(T * k, dtype=torch.int32, device=DEV)
    so = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    moeq.dispatch_mxfp4(tok, torch.from_numpy(ids).to(DEV), out, sf, ro, eids, src, so, slot_rows)
    torch.cuda.synchronize()
    return out, sf, ro, eids, so, rows


def _check_scales(g_sf, ref_sf, ro, so, rows, kv):
    """Logical scale rows of every group's padded range agree."""
    a = L.unswizzle(u8(g_sf), rows, kv)
    b = L.unswizzle(np.asarray(ref_sf), rows, kv)
    for g in range(len(ro) - 1):
        n = (int(ro[g + 1]) - int(ro[g]) + 127) // 128 * 128
        p = int(so[g])
        assert np.array_equal(a[p:p + n], b[p:p + n]), g


@pytest.mark.parametrize("slot_rows", [0, 256])
def test_dispatch_matches_oracle(slot_rows):
    need_gpu()
    moeq.clear_device_error()
    T, H, E, k = 300, 512, 8, 2
    tok = synth.bf16_normal((T, H), 1.0, seed=31, device=DEV, outlier_p=0.01, outlier_scale=40.0)
    ids = _topk(T, k, E, seed=32, zipf=0.8)
    out, sf, ro, eids, so, rows = _dispatch_gpu(tok, ids, E, slot_rows)
    ref = D.dispatch_mxfp4(tok.float().cpu().numpy(), ids, E, max_padded_m=slot_rows,
                           scale_rows_total=rows)
    n = len(ref["src_info"])
    assert np.array_equal(ro.cpu().numpy().view(np.uint32), ref["row_offsets"])
    assert np.array_equal(so.cpu().numpy().view(np.uint32), ref["scales_offsets"])
    assert np.array_equal(u8(out)[:n], ref["q"][:n])
    assert np.all(u8(out)[n:] == 0xA5)
    _check_scales(sf, ref["scales"], ref["row_offsets"], ref["scales_offsets"], rows, H // 32)
    assert moeq.get_device_error() == 0


def test_slot_layout_feeds_the_mxfp4_gemm_like_the_padded_layout():
    need_gpu()
    moeq.clear_device_error()
    T, H, E, k, N = 500, 512, 6, 2, 256
    tok = synth.bf16_normal((T, H), 1.0, seed=41, device=DEV)
    ids = _topk(T, k, E, seed=42, zipf=1.0)
    b = synth.random_fp4_packed((E, N, H // 2), seed=43, device=DEV)
    bsf = synth.random_bytes(E * moeq.sf_bytes(N, H // 32), 116, 126, seed=44, device=DEV)
    res = []
    for slot in (0, 512):
        out, sf, ro, eids, so, rows = _dispatch_gpu(tok, ids, E, slot)
        c = torch.zeros((T * k, N), dtype=torch.bfloat16, device=DEV)
        moeq.grouped_matmul_blockscaled("mxfp4", c, out, sf, b, bsf, None, ro, so, eids, N, H,
                                        rows)
        torch.cuda.synchronize()
        res.append(c)
    assert torch.equal(res[0].view(torch.int16), res[1].view(torch.int16))
    assert (res[0].float().abs() > 0).float().mean() > 0.9
    assert moeq.get_device_error() == 0


def test_slot_overflow_skips_the_group_and_flags_it():
    need_gpu()
    moeq.clear_device_error()
    T, H, E, k = 200, 256, 4, 2
    tok = synth.bf16_normal((T, H), 1.0, seed=51, device=DEV)
    ids = np.zeros((T, k), np.int32)
    ids[:, 0] = 0                     # expert 0 receives 200 rows > one 128-row slot
    ids[:, 1] = 1 + np.arange(T) % 3  # experts 1..3 receive 66-67 rows each
    out, sf, ro, eids, so, rows = _dispatch_gpu(tok, ids, E, slot_rows=128)
    assert moeq.get_device_error() & moeq.DEVERR_SCALE_ROWS
    moeq.clear_device_error()
    ref = D.route_topk(ids, E)
    r = ref[0]
    assert np.array_equal(ro.cpu().numpy().view(np.uint32), r)
    # expert 0's rows are not quantized; experts 1..3 are, as in the oracle
    q = u8(out)
    assert np.all(q[:int(r[1])] == 0xA5)
    x = tok.float().cpu().numpy()[ref[2] // k]
    q_ref, _ = Q.quantize_rows("mxfp4", x[int(r[1]):int(r[4])])
    assert np.array_equal(q[int(r[1]):int(r[4])], q_ref)


def test_dispatch_full_size_sampled():
    """16384 tokens, hidden 4096, top-8 over 128 experts (131072 routed rows):
    the routing exactly, the packed rows and scales of sampled rows."""
    need_gpu()
    moeq.clear_device_error()
    T, H, E, k = 16384, 4096, 128, 8
    tok = synth.bf16_normal((T, H), 1.0, seed=61, device=DEV)
    ids = _topk(T, k, E, seed=62)
    out, sf, ro, eids, so, rows = _dispatch_gpu(tok, ids, E)
    ro_ref, _, src, _ = D.route_topk(ids, E)
    g_ro = ro.cpu().numpy().view(np.uint32)
    assert np.array_equal(g_ro, ro_ref)
    so_ref = Q.padded_scale_offsets(ro_ref)
    assert np.array_equal(so.cpu().numpy().view(np.uint32), so_ref)
    rng = np.random.default_rng(63)
    sample = np.unique(np.concatenate([rng.integers(0, T * k, 200), ro_ref[1:-1] - 1, ro_ref[:-1]]))
    sample = sample[sample < T * k]
    x = tok[torch.from_numpy(src[sample] // k).to(DEV)].float().cpu().numpy()
    q_ref, sc_ref = Q.quantize_rows("mxfp4", x)
    assert np.array_equal(u8(out)[sample], q_ref)
    g = np.searchsorted(ro_ref, sample, side="right") - 1
    srow = so_ref[g] + (sample - ro_ref[g])
    kv = H // 32
    buf = u8(sf)
    cc = np.arange(kv)
    got = buf[L.sf_offset(srow[:, None].astype(np.int64), cc[None, :], kv)]
    assert np.array_equal(got, sc_ref)
    assert moeq.get_device_error() == 0
    note(choices=T * k, sampled_rows=int(len(sample)))


def test_token_level_up_projection_equals_the_row_level_path():
    """Token-major amax, routing, gathered NVFP4 quantization and fused GEMM
    from the tokens and their top-k ids give the bytes of the row-level path
    run on the materialised gathered rows (the two inputs of the benchmark's
    end-to-end figures)."""
    need_gpu()
    moeq.clear_device_error()
    T, K, E, k, I = 300, 512, 8, 4, 192
    tok = synth.bf16_normal((T, K), 1.0, seed=71, device=DEV, outlier_p=0.01, outlier_scale=20.0)
    tk = torch.from_numpy(synth.topk_ids(T, k, E, seed=72, zipf_s=0.7)).to(DEV)
    n = T * k
    rows = moeq.dispatch_scale_rows(T, k, E)
    b = synth.random_fp4_packed((E, 2 * I, K // 2), seed=73, device=DEV)
    bsf = synth.random_bytes(E * moeq.sf_bytes(2 * I, K // 16), 0x18, 0x28, seed=74, device=DEV)
    es = synth.uniform((E,), 0.5, 2.0, seed=75, device=DEV)
    ots = synth.uniform((E,), 0.05, 0.2, seed=76, device=DEV)
    i32 = dict(dtype=torch.int32, device=DEV)
    ro, eids, src, so = (torch.empty(E + 1, **i32), torch.empty(E, **i32), torch.empty(n, **i32),
                         torch.empty(E + 1, **i32))
    moeq.route_topk(tk, ro, eids, src, so)

    def outputs():
        u8z = lambda *shape: torch.zeros(*shape, dtype=torch.uint8, device=DEV)
        return (torch.empty(E, device=DEV), u8z(n, K // 2), u8z(moeq.sf_bytes(rows, K // 16)),
                u8z(n, I // 2), u8z(moeq.sf_bytes(rows, I // 16)))

    ts1, a1, asf1, c1, csf1 = outputs()
    moeq.grouped_amax_scale_topk(tok, tk, ts1, E)
    moeq.grouped_quantize_gather("nvfp4", tok, src, k, a1, asf1, ro, so, eids, ts1, E, rows)
    moeq.grouped_matmul_swiglu(c1, csf1, a1, asf1, b, bsf, es, ots, ro, so, eids, I, K, rows)
    x = tok[torch.div(src, k, rounding_mode="floor").long()].contiguous()
    ts2, a2, asf2, c2, csf2 = outputs()
    moeq.grouped_amax_scale(x, ro, eids, ts2, E)
    moeq.grouped_quantize("nvfp4", x, a2, asf2, ro, so, eids, ts2, E, rows)
    moeq.grouped_matmul_swiglu(c2, csf2, a2, asf2, b, bsf, es, ots, ro, so, eids, I, K, rows)
    torch.cuda.synchronize()
    assert torch.equal(ts1.view(torch.int32), ts2.view(torch.int32))
    assert torch.equal(a1, a2) and torch.equal(asf1, asf2)
    assert torch.equal(c1, c2) and torch.equal(csf1, csf2)
    assert (c1 != 0).float().mean() > 0.3
    assert moeq.get_device_error() == 0


@pytest.mark.parametrize("T,k,E", [(0, 2, 5), (1, 1, 1), (37, 1, 1), (5, 3, 1024)])
def test_route_degenerate_sizes(T, k, E):
    """No tokens, one expert, top-1, more experts than choices."""
    need_gpu()
    moeq.clear_device_error()
    ids = _topk(T, k, E, seed=90 + T) if T else np.zeros((0, k), np.int32)
    ro, eids, src, _ = D.route_topk(ids, E)
    g_ro, g_eids, g_src, g_so = _route_gpu(ids, E)
    assert np.array_equal(g_ro, ro)
    assert np.array_equal(g_eids, eids)
    assert np.array_equal(g_src[:len(src)], src)
    assert np.array_equal(g_so, Q.padded_scale_offsets(ro))
    if T == 0:
        tok = torch.zeros((0, 256), dtype=torch.bfloat16, device=DEV)
        out, sf, ro_d, _, so_d, _ = _dispatch_gpu(tok, ids, E)
        assert int(ro_d[-1]) == 0 and int(so_d[-1]) == 0
    assert moeq.get_device_error() == 0


@pytest.mark.parametrize("T,k,E,K", [(300, 4, 8, 512), (16384, 8, 128, 4096), (100, 40, 64, 256),
                                     (0, 2, 4, 256)])
def test_topk_amax_matches_oracle_and_the_routed_amax(T, k, E, K):
    """Per-expert tensor scales from the tokens and their top-k ids equal the
    oracle's and those of the gathered amax over the routed rows, bit for bit."""
    need_gpu()
    moeq.clear_device_error()
    tok = synth.bf16_normal((T, K), 1.0, seed=81 + T, device=DEV, outlier_p=0.002,
                            outlier_scale=60.0)
    ids = _topk(T, k, E, seed=82) if T else np.zeros((0, k), np.int32)
    tk = torch.from_numpy(ids).to(DEV)
    ts = torch.full((E,), -1.0, device=DEV)
    moeq.grouped_amax_scale_topk(tok, tk, ts, E)
    ref = Q.tensor_scale_from_amax(D.topk_amax(tok.float().cpu().numpy(), ids, E))
    assert np.array_equal(ts.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    if T:
        i32 = dict(dtype=torch.int32, device=DEV)
        ro, eids, src = torch.empty(E + 1, **i32), torch.empty(E, **i32), torch.empty(T * k, **i32)
        moeq.route_topk(tk, ro, eids, src)
        ts2 = torch.empty(E, device=DEV)
        moeq.grouped_amax_scale_gather(tok, src, k, ro, eids, ts2, E)
        assert torch.equal(ts.view(torch.int32), ts2.view(torch.int32))
    assert moeq.get_device_error() == 0


def test_topk_amax_skips_invalid_ids():
    need_gpu()
    moeq.clear_device_error()
    tok = synth.bf16_normal((64, 256), 1.0, seed=91, device=DEV)
    ids = _topk(64, 2, 6, seed=92)
    ids[3, 0] = -2
    ids[40, 1] = 6
    ts = torch.empty(6, device=DEV)
    moeq.grouped_amax_scale_topk(tok, torch.from_numpy(ids).to(DEV), ts, 6)
    ref = Q.tensor_scale_from_amax(D.topk_amax(tok.float().cpu().numpy(), ids, 6))
    assert np.array_equal(ts.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert moeq.get_device_error() & moeq.DEVERR_BAD_EXPERT
    moeq.clear_device_error()


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4", "mxfp8"])
@pytest.mark.parametrize("T,K,E,k,slot_rows", [(600, 1024, 8, 4, 0), (600, 640, 8, 4, 768),
                                               (333, 512, 16, 8, 0), (16384, 4096, 128, 8, 0)])
def test_quantize_topk_equals_the_gathered_quantizer(fmt, T, K, E, k, slot_rows):
    """Token-major quantization (each token read once, written to its routed
    rows) gives the whole output and scale buffers of the gathered quantizer
    byte for byte, canary bytes included; a few choices are dropped."""
    need_gpu()
    moeq.clear_device_error()
    tok = synth.bf16_normal((T, K), 1.0, seed=101 + T, device=DEV, outlier_p=0.003,
                            outlier_scale=40.0)
    ids = _topk(T, k, E, seed=102, zipf=0.9)
    if T < 1000:
        ids[7, 1] = -1
        ids[T - 1, 0] = E
    tk = torch.from_numpy(ids).to(DEV)
    n = T * k
    i32 = dict(dtype=torch.int32, device=DEV)
    ro, eids, src, dst, so = (torch.empty(E + 1, **i32), torch.empty(E, **i32),
                              torch.empty(n, **i32), torch.empty(n, **i32),
                              torch.empty(E + 1, **i32))
    moeq.route_topk(tk, ro, eids, src, so, slot_rows, dst_info=dst)
    ts = torch.empty(E, device=DEV)
    moeq.grouped_amax_scale_topk(tok, tk, ts, E)
    rows = moeq.dispatch_scale_rows(T, k, E, slot_rows)
    ob = K if fmt == "mxfp8" else K // 2
    v = 16 if fmt == "nvfp4" else 32
    outs = []
    for token_major in (True, False):
        out = torch.full((n, ob), 0xA5, dtype=torch.uint8, device=DEV)
        sf = torch.full((moeq.sf_bytes(rows, K // v),), 0x5A, dtype=torch.uint8, device=DEV)
        if token_major:
            moeq.quantize_topk(fmt, tok, tk, dst, out, sf, ro, so, ts, E)
        else:
            moeq.grouped_quantize_gather(fmt, tok, src, k, out, sf, ro, so, eids, ts, E, rows)
        outs.append((out, sf))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])
    routed = int(ro[-1])
    assert (outs[0][0][:routed] != 0xA5).float().mean() > 0.5
    bits = moeq.get_device_error()
    assert (bits & ~moeq.DEVERR_BAD_EXPERT) == 0
    moeq.clear_device_error()
    note(choices=n, routed=routed)
