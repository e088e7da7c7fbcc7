"""Stream order of the library's kernels.  Every kernel is launched with
programmatic stream serialisation, so its CTAs may start while the previous
kernel in the stream finishes; each waits for that kernel's completion before
its first memory access.  Here the whole MoE expert layer (offsets -> amax
-> NVFP4 quantize -> fused gate/up GEMM + SwiGLU + requant -> down-projection
GEMM, and the chained form: block-scaled GEMM -> SwiGLU + requant ->
down-projection) runs three times back to back with no synchronisation, the
intermediate buffers shared by all passes, so every kernel reads what the
one before it wrote and overwrites what an earlier one read.  The outputs
must equal, byte for byte, those of the same calls issued one at a time with
the device synchronised after each -- directly on the stream and replayed
from a captured CUDA graph."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import moeq, synth
from oracle import quantize as Q
from tests._util import DEV, groups_from_counts, need_gpu, to_dev_i32, to_dev_u32

pytestmark = pytest.mark.gpu

E, K, I, H = 8, 512, 256, 256
COUNTS = [0, 1, 127, 129, 260, 3, 64, 200]
PASSES = 3


def _setup():
    ro, ids = groups_from_counts(COUNTS, np.array([3, 0, 7, 1, 5, 2, 6, 4], np.int32))
    so = Q.padded_scale_offsets(ro)
    rows = int(so[-1])
    T = int(ro[-1])
    d = {"T": T, "rows": rows, "ro": to_dev_u32(ro), "ids": to_dev_i32(ids),
         "so": torch.zeros(len(COUNTS) + 1, dtype=torch.int32, device=DEV)}
    d["xs"] = [synth.bf16_normal((T, K), 1.0, seed=10 + i, device=DEV, outlier_p=0.01,
                                 outlier_scale=20.0) for i in range(PASSES)]
    d["b"] = synth.random_fp4_packed((E, 2 * I, K // 2), seed=20, device=DEV)
    d["bsf"] = synth.random_bytes(E * moeq.sf_bytes(2 * I, K // 16), 0x18, 0x28, seed=21, device=DEV)
    d["bd"] = synth.random_fp4_packed((E, H, I // 2), seed=22, device=DEV)
    d["bdsf"] = synth.random_bytes(E * moeq.sf_bytes(H, I // 16), 0x18, 0x28, seed=23, device=DEV)
    d["es"] = synth.uniform((E,), 0.5, 2.0, seed=24, device=DEV)
    d["esd"] = synth.uniform((E,), 0.5, 2.0, seed=25, device=DEV)
    d["ots"] = synth.uniform((E,), 0.05, 0.2, seed=26, device=DEV)
    # intermediates shared by every pass
    d["ts"] = torch.empty(E, dtype=torch.float32, device=DEV)
    d["q"] = torch.empty((T, K // 2), dtype=torch.uint8, device=DEV)
    d["sf"] = torch.empty(moeq.sf_bytes(rows, K // 16), dtype=torch.uint8, device=DEV)
    d["c"] = torch.empty((T, I // 2), dtype=torch.uint8, device=DEV)
    d["csf"] = torch.empty(moeq.sf_bytes(rows, I // 16), dtype=torch.uint8, device=DEV)
    d["y"] = torch.empty((T, 2 * I), dtype=torch.bfloat16, device=DEV)
    d["c2"] = torch.empty_like(d["c"])
    d["csf2"] = torch.empty_like(d["csf"])
    return d


def _scramble(d):
    for k in ("so", "ts", "q", "sf", "c", "csf", "y", "c2", "csf2"):
        d[k].view(torch.uint8).fill_(0xA7)


def _pass(d, i, out, out2, sync):
    def step():
        if sync:
            torch.cuda.synchronize()
    r, T = d["rows"], d["T"]
    moeq.padded_scale_offsets(d["ro"], d["so"]); step()
    moeq.grouped_amax_scale(d["xs"][i], d["ro"], d["ids"], d["ts"], E); step()
    moeq.grouped_quantize("nvfp4", d["xs"][i], d["q"], d["sf"], d["ro"], d["so"], d["ids"],
                          d["ts"], E, r); step()
    moeq.grouped_matmul_swiglu(d["c"], d["csf"], d["q"], d["sf"], d["b"], d["bsf"], d["es"],
                               d["ots"], d["ro"], d["so"], d["ids"], I, K, r); step()
    moeq.grouped_matmul_blockscaled("nvfp4", out, d["c"], d["csf"], d["bd"], d["bdsf"], d["esd"],
                                    d["ro"], d["so"], d["ids"], H, I, r); step()
    moeq.grouped_matmul_blockscaled("nvfp4", d["y"], d["q"], d["sf"], d["b"], d["bsf"], d["es"],
                                    d["ro"], d["so"], d["ids"], 2 * I, K, r); step()
    moeq.swiglu_quantize(d["c2"], d["csf2"], d["y"], d["ots"], d["ro"], d["so"], d["ids"], E,
                         r); step()
    moeq.grouped_matmul_blockscaled("nvfp4", out2, d["c2"], d["csf2"], d["bd"], d["bdsf"],
                                    d["esd"], d["ro"], d["so"], d["ids"], H, I, r); step()


def _outs(d):
    return ([torch.zeros((d["T"], H), dtype=torch.bfloat16, device=DEV) for _ in range(PASSES)],
            [torch.zeros((d["T"], H), dtype=torch.bfloat16, device=DEV) for _ in range(PASSES)])


def _bits(t):
    return t.view(torch.int16)


def test_back_to_back_layers_equal_synchronised_calls():
    need_gpu()
    moeq.clear_device_error()
    d = _setup()
    ref, ref2 = _outs(d)
    for i in range(PASSES):
        _pass(d, i, ref[i], ref2[i], sync=True)
    # the fused and the chained layer agree, and the passes differ
    for i in range(PASSES):
        assert torch.equal(_bits(ref[i]), _bits(ref2[i]))
        assert (ref[i].float().abs() > 0).float().mean() > 0.5
    assert not torch.equal(_bits(ref[0]), _bits(ref[1]))

    _scramble(d)
    got, got2 = _outs(d)
    for i in range(PASSES):
        _pass(d, i, got[i], got2[i], sync=False)
    torch.cuda.synchronize()
    for i in range(PASSES):
        assert torch.equal(_bits(got[i]), _bits(ref[i])), i
        assert torch.equal(_bits(got2[i]), _bits(ref2[i])), i
    assert moeq.get_device_error() == 0


def test_graph_replay_equals_synchronised_calls():
    need_gpu()
    moeq.clear_device_error()
    d = _setup()
    ref, ref2 = _outs(d)
    for i in range(PASSES):
        _pass(d, i, ref[i], ref2[i], sync=True)
    got, got2 = _outs(d)
    # warm the per-device launch set-up outside the capture
    _pass(d, 0, got[0], got2[0], sync=False)
    torch.cuda.synchronize()
    _scramble(d)
    for t in got + got2:
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(PASSES):
            _pass(d, i, got[i], got2[i], sync=False)
    for _ in range(2):
        _scramble(d)
        for t in got + got2:
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for i in range(PASSES):
            assert torch.equal(_bits(got[i]), _bits(ref[i])), i
            assert torch.equal(_bits(got2[i]), _bits(ref2[i])), i
    assert moeq.get_device_error() == 0
