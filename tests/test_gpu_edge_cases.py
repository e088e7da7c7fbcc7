"""Edge cases of the grouped path at the limits of its tables and shapes,
against the CPU oracle through the C ABI:
* the quantizer with more groups than its shared-memory group table (the
  global-memory lookup path), all three formats, bit-exact;
* the grouped GEMMs at the scheduler's maximum of 1024 groups (most of them
  empty or 1-8 rows, expert ids repeating), FP8 rowwise and NVFP4;
* a long reduction (K = 16384) in the block-scaled GEMM;
* the fused SwiGLU kernels (NVFP4 and MXFP4) byte-identical to the chained
  path at 512 groups (silu from the kernel's shared-memory table) and at 513
  and 1024 groups (silu computed: the table's launches hold at most 512)."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import moeq, synth
from oracle import gemm as OG
from oracle import layout as L
from oracle import quantize as Q
from tests._util import (DEV, assert_gemm_close, bf16_bits, groups_from_counts, need_gpu,
                         to_dev_i32, to_dev_u32, u8)
from tests.test_gpu_gemm import CANARY, blockscaled_inputs, run_blockscaled

pytestmark = pytest.mark.gpu


def _many_groups(G, E, seed, max_rows=8):
    rng = np.random.default_rng(seed)
    counts = rng.integers(0, max_rows + 1, G)
    counts[rng.random(G) < 0.4] = 0
    counts[G // 2] = 300                                  # one multi-tile group
    ids = rng.integers(0, E, G).astype(np.int32)
    return groups_from_counts(counts, ids)


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp8", "mxfp4"])
def test_quantize_more_groups_than_the_shared_table(fmt):
    need_gpu()
    G, E, K = 700, 64, 256
    ro, ids = _many_groups(G, E, seed=1)
    so = Q.padded_scale_offsets(ro)
    T, rows = int(ro[-1]) + 3, int(so[-1]) + 128
    x = synth.bf16_normal((T, K), 1.0, seed=2, outlier_p=0.01, outlier_scale=20.0)
    x_np = x.float().numpy()
    ts = Q.tensor_scale_from_amax(Q.group_amax(x_np, ro, ids, E))
    v = 16 if fmt == "nvfp4" else 32
    ob = K if fmt == "mxfp8" else K // 2
    out = torch.full((T, ob), 0xA5, dtype=torch.uint8, device=DEV)
    sf = torch.full((moeq.sf_bytes(rows, K // v),), 0x5A, dtype=torch.uint8, device=DEV)
    amax = torch.empty(E, device=DEV)
    moeq.grouped_amax_scale(x.to(DEV), to_dev_u32(ro), to_dev_i32(ids), amax, E)
    moeq.grouped_quantize(fmt, x.to(DEV), out, sf, to_dev_u32(ro), to_dev_u32(so),
                          to_dev_i32(ids), amax, E, rows)
    torch.cuda.synchronize()
    assert np.array_equal(amax.cpu().numpy().view(np.uint32), ts.view(np.uint32))
    want_out, want_sf = Q.grouped_quantize(fmt, x_np, ro, so, ids, ts,
                                           out=np.full((T, ob), 0xA5, np.uint8),
                                           scales=np.full(L.physical_bytes(rows, K // v), 0x5A,
                                                          np.uint8), scale_rows_total=rows)
    assert np.array_equal(u8(out), want_out) and np.array_equal(u8(sf), want_sf)
    assert moeq.get_device_error() == 0


def test_rowwise_fp8_max_groups():
    need_gpu()
    G, E, N, K = 1024, 96, 256, 256
    ro, ids = _many_groups(G, E, seed=3)
    T = int(ro[-1]) + 4
    a = synth.e4m3_normal((T, K), 1.0, seed=4)
    b = synth.e4m3_normal((E, N, K), 0.5, seed=5)
    sa = synth.uniform((T,), 0.01, 0.1, seed=6)
    sb = synth.uniform((E, N), 0.005, 0.05, seed=7)
    c = torch.full((T, N), CANARY, dtype=torch.bfloat16, device=DEV)
    moeq.grouped_matmul_rowwise_fp8(c, a.to(DEV), b.to(DEV), sa.to(DEV), sb.to(DEV),
                                    to_dev_u32(ro), to_dev_i32(ids))
    torch.cuda.synchronize()
    out = bf16_bits(c)
    _, f64 = OG.grouped_matmul_rowwise_fp8(u8(a), u8(b), sa.numpy(), sb.numpy(), ro, ids,
                                           return_f64=True)
    written = np.zeros(T, bool)
    written[:int(ro[-1])] = True
    assert_gemm_close(out, f64, mask_rows=written)
    assert np.all(out[~written] == np.float32(CANARY).view(np.uint32) >> 16)


@pytest.mark.parametrize("G,K", [(1024, 256), (5, 16384)])
def test_nvfp4_blockscaled_max_groups_and_long_k(G, K):
    need_gpu()
    E, N = 96, 256
    if G == 5:
        ro, ids = groups_from_counts([40, 0, 129, 7, 200], [3, 1, 0, 2, 4])
    else:
        ro, ids = _many_groups(G, E, seed=8)
    so = Q.padded_scale_offsets(ro)
    T, rows = int(ro[-1]) + 2, int(so[-1]) + 128
    a, asf, b, bsf, es = blockscaled_inputs("nvfp4", T, E, N, K, rows, seed=9)
    c = bf16_bits(run_blockscaled("nvfp4", a, asf, b, bsf, es, ro, so, ids, N, K, rows))
    _, f64 = OG.grouped_matmul_blockscaled("nvfp4", u8(a), u8(asf), u8(b), u8(bsf), es.numpy(),
                                           ro, so, ids, N=N, K=K, scale_rows_total=rows,
                                           return_f64=True)
    written = np.zeros(T, bool)
    written[:int(ro[-1])] = True
    assert_gemm_close(c, f64, mask_rows=written)
    assert np.all(c[~written] == np.float32(CANARY).view(np.uint32) >> 16)


@pytest.mark.parametrize("fmt,G", [("nvfp4", 512), ("nvfp4", 513), ("nvfp4", 1024),
                                   ("mxfp4", 512), ("mxfp4", 513)])
def test_fused_swiglu_many_groups_equals_chained(fmt, G):
    need_gpu()
    E, I, K = 96, 128, 256
    ro, ids = _many_groups(G, E, seed=10)
    so = Q.padded_scale_offsets(ro)
    T, rows = int(ro[-1]) + 2, int(so[-1]) + 128
    a, asf, b, bsf, es = blockscaled_inputs(fmt, T, E, 2 * I, K, rows, seed=11, device=DEV)
    ro_d, so_d, ids_d = to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids)
    y = torch.zeros((T, 2 * I), dtype=torch.bfloat16, device=DEV)
    moeq.grouped_matmul_blockscaled(fmt, y, a, asf, b, bsf, es, ro_d, so_d, ids_d, 2 * I, K,
                                    rows)
    if fmt == "nvfp4":
        ots = synth.uniform((E,), 0.05, 0.2, seed=12, device=DEV)
        c1 = torch.full((T, I // 2), 0xA5, dtype=torch.uint8, device=DEV)
        s1 = torch.full((moeq.sf_bytes(rows, I // 16),), 0x5A, dtype=torch.uint8, device=DEV)
        moeq.swiglu_quantize(c1, s1, y, ots, ro_d, so_d, ids_d, E, rows)
        c2, s2 = torch.full_like(c1, 0xA5), torch.full_like(s1, 0x5A)
        moeq.grouped_matmul_swiglu(c2, s2, a, asf, b, bsf, es, ots, ro_d, so_d, ids_d, I, K, rows)
    else:
        c1 = torch.full((T, I // 2), 0xA5, dtype=torch.uint8, device=DEV)
        s1 = torch.full((moeq.sf_bytes(rows, I // 32),), 0x5A, dtype=torch.uint8, device=DEV)
        moeq.swiglu_quantize_mx(fmt, c1, s1, y, ro_d, so_d, ids_d, E, rows)
        c2, s2 = torch.full_like(c1, 0xA5), torch.full_like(s1, 0x5A)
        moeq.grouped_matmul_swiglu_mx(fmt, c2, s2, a, asf, b, bsf, es, ro_d, so_d, ids_d, I, K,
                                      rows)
    torch.cuda.synchronize()
    assert torch.equal(c1, c2) and torch.equal(s1, s2)
    assert (c1[:int(ro[-1])] != 0).float().mean() > 0.3
    assert moeq.get_device_error() == 0
