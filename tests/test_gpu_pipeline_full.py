"""The NVFP4 up-projection at full size, with inputs made as the 128-expert
workload describes them: activations bf16 N(0, 1) and gate/up weights bf16
N(0, 0.02) ([128, 2 x 1536, 4096], gate/up interleaved), both quantized to
NVFP4 by the library's grouped quantizer with per-expert tensor scales from
their amax, expert scales U[0.5, 2].

Checks ("max.nn.moe.NvMxf4f8Strategy": grouped_quantize, grouped_matmul,
grouped_matmul_swiglu; "grouped_quantize_dynamic_scaled_fp4_async_kernel"):
* fused GEMM + SwiGLU + requant equals the chained path, whole buffers;
* on rows of the first, middle and last m-block of every group and on four
  32-column output blocks per expert (spread over the n-tiles), the oracle,
  working from the seeded bf16 tensors alone: the quantized activation and
  weight rows and their scales bit-exact, the chained GEMM's y within the
  GEMM tolerance, and the fused output's codes and scales bit-exact on every
  block where the oracle's bf16 y equals the GPU's (the fp32 accumulation
  order is the kernel's; the rest of the chain is fixed operation by
  operation).

The SwiGLU output tensor scale of each expert is taken from the oracle's own
h on the sampled points (amax x 4 / 2688), so that no oracle input comes
from the GPU."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import moeq, synth
from oracle import formats as F
from oracle import gemm as OG
from oracle import layout as L
from oracle import quantize as Q
from oracle import swiglu as S
from tests._util import (DEV, assert_gemm_close, bf16_bits, group_sample_rows, need_gpu, note,
                         to_dev_i32, to_dev_u32, u8)

pytestmark = pytest.mark.gpu

E, TOKENS, TOPK, K, I = 128, 16384, 8, 4096, 1536
N = 2 * I


def _expert_blocks(e):
    """Four 32-column output blocks (16 SwiGLU outputs each) of expert e:
    the first, the last and two that move with e across the n-tiles."""
    nblk = N // 32
    return sorted({0, (7 * e + 3) % nblk, nblk // 2 + e % (nblk // 2), nblk - 1})


def _rows_u8(t, rows):
    t = t if t.dtype == torch.uint8 else t.view(torch.uint8)
    return u8(t.index_select(0, torch.from_numpy(np.asarray(rows, np.int64)).to(t.device)))


def test_up_projection_recipe_full_size():
    need_gpu()
    counts = synth.routing_counts(TOKENS, TOPK, E, seed=0)
    ro, ids = synth.ragged_groups(counts)
    so = Q.padded_scale_offsets(ro)
    T, rows_total = int(ro[-1]), int(so[-1])
    x = synth.bf16_normal((T, K), 1.0, seed=81, device=DEV)
    w = synth.bf16_normal((E * N, K), 0.02, seed=82, device=DEV)
    es = synth.uniform((E,), 0.5, 2.0, seed=83)
    kv = K // 16

    # ---- GPU: quantize weights (one group per expert) and activations
    w_offs = np.arange(E + 1, dtype=np.uint32) * N
    w_ids = np.arange(E, dtype=np.int32)
    ts_w = torch.empty(E, device=DEV)
    moeq.grouped_amax_scale(w, to_dev_u32(w_offs), to_dev_i32(w_ids), ts_w, E)
    b = torch.empty((E * N, K // 2), dtype=torch.uint8, device=DEV)
    bsf = torch.empty(moeq.sf_bytes(E * N, kv), dtype=torch.uint8, device=DEV)
    moeq.grouped_quantize("nvfp4", w, b, bsf, to_dev_u32(w_offs), to_dev_u32(w_offs),
                          to_dev_i32(w_ids), ts_w, E, E * N, N)
    ro_d, so_d, ids_d = to_dev_u32(ro), to_dev_u32(so), to_dev_i32(ids)
    ts_a = torch.empty(E, device=DEV)
    moeq.grouped_amax_scale(x, ro_d, ids_d, ts_a, E)
    a = torch.empty((T, K // 2), dtype=torch.uint8, device=DEV)
    asf = torch.empty(moeq.sf_bytes(rows_total, kv), dtype=torch.uint8, device=DEV)
    moeq.grouped_quantize("nvfp4", x, a, asf, ro_d, so_d, ids_d, ts_a, E, rows_total,
                          int(counts.max()))
    torch.cuda.synchronize()

    # ---- oracle: tensor scales from the seeded bf16 tensors
    x_cpu = x.cpu()
    amax_a = np.zeros(E, np.float32)
    for g in range(len(ids)):
        r0, r1 = int(ro[g]), int(ro[g + 1])
        if r1 > r0:
            amax_a[ids[g]] = max(amax_a[ids[g]],
                                 float(x_cpu[r0:r1].float().abs().max()))
    ts_a_o = Q.tensor_scale_from_amax(amax_a)
    assert np.array_equal(ts_a.cpu().numpy().view(np.uint32), ts_a_o.view(np.uint32))
    w_cpu = w.cpu()
    amax_w = np.array([float(w_cpu[e * N:(e + 1) * N].float().abs().max()) for e in range(E)],
                      np.float32)
    ts_w_o = Q.tensor_scale_from_amax(amax_w)
    assert np.array_equal(ts_w.cpu().numpy().view(np.uint32), ts_w_o.view(np.uint32))

    # ---- oracle: quantized sampled rows, GEMM, SwiGLU on the sampled points
    sample = group_sample_rows(ro)
    asf_np, bsf_np = u8(asf), u8(bsf)
    kcols = np.arange(kv)[None, :]
    per_group = []
    for g, rows in enumerate(sample):
        if rows.size == 0:
            continue
        e = int(ids[g])
        blocks = _expert_blocks(e)
        cols = np.concatenate([np.arange(32 * j, 32 * j + 32) for j in blocks])
        # activations: codes and scales bit-exact
        qa, sa = Q.quantize_rows("nvfp4", x_cpu[torch.from_numpy(rows)].float().numpy(),
                                 ts_a_o[e])
        prow = int(so[g]) + rows - int(ro[g])
        assert np.array_equal(_rows_u8(a, rows), qa)
        assert np.array_equal(asf_np[L.sf_offset(prow[:, None], kcols, kv)], sa)
        # weights (the sampled gate/up rows of expert e): bit-exact
        wrow = e * N + cols
        qb, sb = Q.quantize_rows("nvfp4", w_cpu[torch.from_numpy(wrow)].float().numpy(),
                                 ts_w_o[e])
        assert np.array_equal(_rows_u8(b, wrow), qb)
        assert np.array_equal(bsf_np[L.sf_offset(wrow[:, None], kcols, kv)], sb)
        # GEMM from the oracle's own operands
        pad = np.zeros((128, kv), np.uint8)
        pad[:len(rows)] = sa
        _, f64 = OG.grouped_matmul_blockscaled(
            "nvfp4", qa, L.swizzle(pad), qb[None], L.swizzle(sb), es.numpy()[e:e + 1],
            np.array([0, len(rows)], np.uint32), np.array([0, 128], np.uint32), [0],
            N=len(cols), K=K, scale_rows_total=128, return_f64=True)
        y_o = F.decode_bf16(F.encode_bf16(f64))          # the oracle's bf16 y
        per_group.append((g, e, rows, prow, blocks, cols, f64, y_o))

    # output scales from the oracle's h on the sampled points (x 4 margin)
    hmax = np.zeros(E, np.float32)
    for g, e, rows, prow, blocks, cols, f64, y_o in per_group:
        hmax[e] = max(hmax[e], float(np.abs(S.swiglu(y_o.astype(np.float32))).max()))
    ots = np.where(hmax > 0, (hmax * np.float32(4.0)) / np.float32(2688.0),
                   np.float32(1.0)).astype(np.float32)

    # ---- GPU: chained (bf16 y -> SwiGLU + requant) and fused
    y = torch.empty((T, N), dtype=torch.bfloat16, device=DEV)
    b3 = b.view(E, N, K // 2)
    es_d, ots_d = es.to(DEV), torch.from_numpy(ots).to(DEV)
    moeq.grouped_matmul_blockscaled("nvfp4", y, a, asf, b3, bsf, es_d, ro_d, so_d, ids_d, N, K,
                                    rows_total, int(counts.max()))
    c1 = torch.full((T, I // 2), 0xA5, dtype=torch.uint8, device=DEV)
    s1 = torch.full((moeq.sf_bytes(rows_total, I // 16),), 0x5A, dtype=torch.uint8, device=DEV)
    moeq.swiglu_quantize(c1, s1, y, ots_d, ro_d, so_d, ids_d, E, rows_total, int(counts.max()))
    c2 = torch.full_like(c1, 0xA5)
    s2 = torch.full_like(s1, 0x5A)
    moeq.grouped_matmul_swiglu(c2, s2, a, asf, b3, bsf, es_d, ots_d, ro_d, so_d, ids_d, I, K,
                               rows_total, int(counts.max()))
    torch.cuda.synchronize()
    assert moeq.get_device_error() == 0
    assert torch.equal(c1, c2) and torch.equal(s1, s2)

    # ---- GPU vs oracle on the sampled points
    c_np, s_np = u8(c2), u8(s2)
    checked = total = 0
    for g, e, rows, prow, blocks, cols, f64, y_o in per_group:
        yg = bf16_bits(y.index_select(0, torch.from_numpy(rows).to(DEV)))[:, cols]
        assert_gemm_close(yg, f64)
        y_gpu = F.decode_bf16(yg)
        for bi, j in enumerate(blocks):
            sl = slice(32 * bi, 32 * bi + 32)
            h = S.swiglu(y_o[:, sl].astype(np.float32))              # [rows, 16]
            q, sc = Q.quantize_rows("nvfp4", h, ots[e])
            same = np.all(y_gpu[:, sl] == y_o[:, sl], axis=1)
            total += len(rows)
            for i in np.nonzero(same)[0]:
                assert np.array_equal(c_np[rows[i], 8 * j:8 * j + 8], q[i])
                off = L.sf_offset(prow[i], j, I // 16)
                assert s_np[off] == sc[i, 0]
                checked += 1
    note(requant_blocks_checked=checked, requant_blocks_sampled=total)
    assert checked >= 0.5 * total
