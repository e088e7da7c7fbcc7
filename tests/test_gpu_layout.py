"""GPU parity of the weight-preparation layout calls, through the C ABI:
logical <-> tiled block-scale layout and the gate/up row interleave are
byte-exact against the oracle's index function; and preparing an NVFP4
gate/up weight from separately quantized gate and up halves gives exactly
the bytes of quantizing the interleaved weight in one call."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import moeq, synth
from oracle import layout as L
from tests._util import DEV, need_gpu, to_dev_i32, to_dev_u32, u8

pytestmark = pytest.mark.gpu


def _rand_u8(shape, seed):
    return np.random.default_rng(seed).integers(0, 256, shape, dtype=np.uint8)


@pytest.mark.parametrize("batch,rows,kv", [(1, 128, 4), (3, 200, 10), (2, 3072, 256),
                                           (1, 1, 1), (5, 129, 96)])
def test_sf_swizzle_and_unswizzle(batch, rows, kv):
    need_gpu()
    logical = _rand_u8((batch, rows, kv), seed=rows * kv + batch)
    tiled = torch.full((batch * moeq.sf_bytes(rows, kv),), 0x77, dtype=torch.uint8, device=DEV)
    moeq.sf_swizzle(tiled, torch.from_numpy(logical).to(DEV))
    torch.cuda.synchronize()
    got = u8(tiled).reshape(batch, -1)
    for b in range(batch):
        assert np.array_equal(got[b], L.swizzle(logical[b]))   # padding bytes written 0
    back = torch.full((batch, rows, kv), 0x33, dtype=torch.uint8, device=DEV)
    moeq.sf_unswizzle(back, tiled)
    torch.cuda.synchronize()
    assert np.array_equal(u8(back), logical)


@pytest.mark.parametrize("rows,row_bytes", [(3, 2048), (17, 7), (64, 96)])
def test_interleave_gate_up(rows, row_bytes):
    need_gpu()
    gate = _rand_u8((4, rows, row_bytes), seed=rows)
    up = _rand_u8((4, rows, row_bytes), seed=rows + 1)
    out = torch.full((4, 2 * rows, row_bytes), 0x11, dtype=torch.uint8, device=DEV)
    moeq.interleave_gate_up(out, torch.from_numpy(gate).to(DEV), torch.from_numpy(up).to(DEV))
    torch.cuda.synchronize()
    assert np.array_equal(u8(out), L.interleave_rows(gate, up))


def _quantize_weight(w, ts):
    """NVFP4 of bf16 weights [E, R, K] with per-expert tensor scales ts,
    one group of R rows per expert (R % 128 == 0: no padding rows)."""
    E, R, K = w.shape
    ro = to_dev_u32(np.arange(E + 1, dtype=np.uint32) * R)
    so = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    moeq.padded_scale_offsets(ro, so)
    q = torch.empty((E * R, K // 2), dtype=torch.uint8, device=DEV)
    sf = torch.empty(moeq.sf_bytes(E * R, K // 16), dtype=torch.uint8, device=DEV)
    moeq.grouped_quantize("nvfp4", w.reshape(E * R, K), q, sf, ro, so,
                          to_dev_i32(np.arange(E)), ts, E, E * R, R)
    return q.reshape(E, R, K // 2), sf


def test_prepared_gate_up_weight_equals_interleaved_quantization():
    need_gpu()
    E, I, K = 3, 256, 512
    gate = synth.bf16_normal((E, I, K), 0.02, seed=90, device=DEV)
    up = synth.bf16_normal((E, I, K), 0.02, seed=91, device=DEV)
    ts = synth.uniform((E,), 1e-5, 3e-5, seed=92, device=DEV)
    # the reference: quantize the interleaved bf16 weight in one call
    inter = torch.empty((E, 2 * I, K), dtype=torch.bfloat16, device=DEV)
    inter[:, 0::2] = gate
    inter[:, 1::2] = up
    q_ref, sf_ref = _quantize_weight(inter, ts)
    # prepared: gate and up quantized separately, then interleaved
    qg, sfg = _quantize_weight(gate, ts)
    qu, sfu = _quantize_weight(up, ts)
    q = torch.empty_like(q_ref)
    moeq.interleave_gate_up(q, qg, qu)
    kv = K // 16
    lg = torch.empty((E, I, kv), dtype=torch.uint8, device=DEV)
    lu = torch.empty_like(lg)
    moeq.sf_unswizzle(lg, sfg)
    moeq.sf_unswizzle(lu, sfu)
    li = torch.empty((E, 2 * I, kv), dtype=torch.uint8, device=DEV)
    moeq.interleave_gate_up(li, lg, lu)
    sf = torch.empty_like(sf_ref)
    moeq.sf_swizzle(sf, li)
    torch.cuda.synchronize()
    assert torch.equal(q, q_ref)
    assert torch.equal(sf, sf_ref)
    assert moeq.get_device_error() == 0
