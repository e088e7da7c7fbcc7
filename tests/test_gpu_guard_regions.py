"""Guard regions around every output buffer.  Each output of every entry
point is a view into a larger buffer filled with a canary byte, with 4 KB of
canary before and after it; after the call (ragged groups: empty groups,
groups of 1 / 127 / 129 rows, rows past the last group, N not a multiple of
the 256-column tile) both guards must still hold only the canary.  The
parity tests check the bytes inside the buffers; this checks that nothing is
written outside them."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import moeq, synth
from oracle import quantize as Q
from tests._util import DEV, groups_from_counts, need_gpu, note, to_dev_i32, to_dev_u32
from tests.test_gpu_gemm import blockscaled_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096
FILL = 0xA5
COUNTS = [0, 1, 127, 129, 3, 200]
IDS = [4, 0, 2, 5, 1, 3]
E = 6
TAIL = 5            # rows after the last group, inside the buffers


class Guarded:
    """Output tensors carved out of canary-filled buffers with guards."""

    def __init__(self):
        self.items = []

    def __call__(self, shape, dtype):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        back = torch.full((GUARD + n + GUARD,), FILL, dtype=torch.uint8, device=DEV)
        self.items.append((back, n))
        return back[GUARD:GUARD + n].view(dtype).view(*shape)

    def check(self):
        torch.cuda.synchronize()
        for i, (back, n) in enumerate(self.items):
            assert bool((back[:GUARD] == FILL).all()), f"output {i}: write before its buffer"
            assert bool((back[GUARD + n:] == FILL).all()), f"output {i}: write past its buffer"
        note(guarded_outputs=len(self.items))


def _groups():
    ro, ids = groups_from_counts(COUNTS, np.array(IDS, np.int32))
    so = Q.padded_scale_offsets(ro)
    return ro, ids, so, int(so[-1]), int(ro[-1]) + TAIL


def test_quantizer_entry_points_stay_in_their_buffers():
    need_gpu()
    moeq.clear_device_error()
    ro, ids, so, rows, T = _groups()
    K = 1024
    g = Guarded()
    ro_d, ids_d = to_dev_u32(ro), to_dev_i32(ids)
    so_d = g((len(ids) + 1,), torch.int32)
    moeq.padded_scale_offsets(ro_d, so_d)
    x = synth.bf16_normal((T, K), 1.0, seed=3, device=DEV, outlier_p=0.01, outlier_scale=30.0)
    ts = g((E,), torch.float32)
    moeq.grouped_amax_scale(x, ro_d, ids_d, ts, E)
    for fmt, ob, v in (("nvfp4", K // 2, 16), ("mxfp4", K // 2, 32), ("mxfp8", K, 32)):
        q = g((T, ob), torch.uint8)
        sf = g((moeq.sf_bytes(rows, K // v),), torch.uint8)
        moeq.grouped_quantize(fmt, x, q, sf, ro_d, so_d, ids_d, ts, E, rows)
    # gathered rows: row t of the output reads input row idx[t] // 2
    idx = torch.from_numpy(np.random.default_rng(4).integers(0, 2 * T, T).astype(np.int32)).to(DEV)
    ts2 = g((E,), torch.float32)
    moeq.grouped_amax_scale_gather(x, idx, 2, ro_d, ids_d, ts2, E)
    q = g((T, K // 2), torch.uint8)
    sf = g((moeq.sf_bytes(rows, K // 16),), torch.uint8)
    moeq.grouped_quantize_gather("nvfp4", x, idx, 2, q, sf, ro_d, so_d, ids_d, ts2, E, rows)
    g.check()
    assert moeq.get_device_error() == 0


def test_gemm_entry_points_stay_in_their_buffers():
    need_gpu()
    moeq.clear_device_error()
    ro, ids, so, rows, T = _groups()
    ro_d, ids_d, so_d = to_dev_u32(ro), to_dev_i32(ids), to_dev_u32(so)
    g = Guarded()
    # FP8 rowwise, N = 384 (one full and one half 256-column tile), and N = 64
    for N in (384, 64):
        K = 256
        a = synth.e4m3_normal((T, K), 1.0, seed=5, device=DEV)
        b = synth.e4m3_normal((E, N, K), 0.5, seed=6, device=DEV)
        sa = synth.uniform((T,), 0.01, 0.1, seed=7, device=DEV)
        sb = synth.uniform((E, N), 0.005, 0.05, seed=8, device=DEV)
        c = g((T, N), torch.bfloat16)
        moeq.grouped_matmul_rowwise_fp8(c, a, b, sa, sb, ro_d, ids_d)
    # block-scaled, bf16 out, N = 384
    N, K = 384, 512
    for fmt in ("nvfp4", "mxfp4", "mxfp8"):
        a, asf, b, bsf, es = blockscaled_inputs(fmt, T, E, N, K, rows, seed=11, device=DEV)
        c = g((T, N), torch.bfloat16)
        moeq.grouped_matmul_blockscaled(fmt, c, a, asf, b, bsf, es, ro_d, so_d, ids_d, N, K, rows)
    # fused gate/up GEMM + SwiGLU + requant, I = 192 (2I = 384)
    I = 192
    ots = synth.uniform((E,), 0.05, 0.2, seed=12, device=DEV)
    a, asf, b, bsf, es = blockscaled_inputs("nvfp4", T, E, 2 * I, K, rows, seed=13, device=DEV)
    c = g((T, I // 2), torch.uint8)
    csf = g((moeq.sf_bytes(rows, I // 16),), torch.uint8)
    moeq.grouped_matmul_swiglu(c, csf, a, asf, b, bsf, es, ots, ro_d, so_d, ids_d, I, K, rows)
    I = 256   # MX outputs need I a multiple of 128
    for fmt in ("mxfp4", "mxfp8"):
        a, asf, b, bsf, es = blockscaled_inputs(fmt, T, E, 2 * I, K, rows, seed=14, device=DEV)
        c = g((T, I if fmt == "mxfp8" else I // 2), torch.uint8)
        csf = g((moeq.sf_bytes(rows, I // 32),), torch.uint8)
        moeq.grouped_matmul_swiglu_mx(fmt, c, csf, a, asf, b, bsf, es, ro_d, so_d, ids_d, I, K,
                                      rows)
    g.check()
    assert moeq.get_device_error() == 0


def test_swiglu_and_layout_entry_points_stay_in_their_buffers():
    need_gpu()
    moeq.clear_device_error()
    ro, ids, so, rows, T = _groups()
    ro_d, ids_d, so_d = to_dev_u32(ro), to_dev_i32(ids), to_dev_u32(so)
    g = Guarded()
    I = 256
    y = synth.bf16_normal((T, 2 * I), 1.0, seed=21, device=DEV)
    ots = synth.uniform((E,), 0.05, 0.2, seed=22, device=DEV)
    c = g((T, I // 2), torch.uint8)
    csf = g((moeq.sf_bytes(rows, I // 16),), torch.uint8)
    moeq.swiglu_quantize(c, csf, y, ots, ro_d, so_d, ids_d, E, rows)
    for fmt in ("mxfp4", "mxfp8"):
        c = g((T, I if fmt == "mxfp8" else I // 2), torch.uint8)
        csf = g((moeq.sf_bytes(rows, I // 32),), torch.uint8)
        moeq.swiglu_quantize_mx(fmt, c, csf, y, ro_d, so_d, ids_d, E, rows)
    # scale layout helpers (rows and kv not multiples of the 128 x 4 atom)
    logical = synth.random_bytes(3 * 130 * 9, 0, 255, seed=23, device=DEV).view(3, 130, 9)
    tiled = g((3 * moeq.sf_bytes(130, 9),), torch.uint8)
    moeq.sf_swizzle(tiled, logical)
    back = g((3, 130, 9), torch.uint8)
    moeq.sf_unswizzle(back, tiled)
    assert torch.equal(back, logical)
    gate = synth.random_bytes(2 * 7 * 24, 0, 255, seed=24, device=DEV).view(2, 7, 24)
    up = synth.random_bytes(2 * 7 * 24, 0, 255, seed=25, device=DEV).view(2, 7, 24)
    out = g((2, 14, 24), torch.uint8)
    moeq.interleave_gate_up(out, gate, up)
    g.check()
    assert moeq.get_device_error() == 0


def test_dispatch_entry_points_stay_in_their_buffers():
    need_gpu()
    moeq.clear_device_error()
    T, H, E, k = 300, 256, 7, 3
    g = Guarded()
    tok = synth.bf16_normal((T, H), 1.0, seed=31, device=DEV)
    ids = torch.from_numpy(synth.topk_ids(T, k, E, seed=32, zipf_s=1.0)).to(DEV)
    for slot in (0, 384):
        ro = g((E + 1,), torch.int32)
        eids = g((E,), torch.int32)
        src = g((T * k,), torch.int32)
        so = g((E + 1,), torch.int32)
        moeq.route_topk(ids, ro, eids, src, so, slot)
        rows = moeq.dispatch_scale_rows(T, k, E, slot)
        out = g((T * k, H // 2), torch.uint8)
        sf = g((moeq.sf_bytes(rows, H // 32),), torch.uint8)
        moeq.dispatch_mxfp4(tok, ids, out, sf, ro, eids, src, so, slot)
    ts = g((E,), torch.float32)
    moeq.grouped_amax_scale_topk(tok, ids, ts, E)
    g.check()
    assert moeq.get_device_error() == 0
