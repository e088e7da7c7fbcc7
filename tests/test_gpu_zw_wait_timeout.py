"""Failure detection on the GPU without a fault: a test build of the library
(MOEQ_TEST_STUCK_STAGE) announces the first pipeline stage of every CTA's
first tile on its barrier but never loads it, so the bounded waits on that
barrier run out (about a second).  The kernel must then set the sticky
timeout bit, let every other role leave its loop, let every copy it
announced land, free tensor memory and exit; the host reads the bit through
moeq_get_device_error, and the same context keeps working.  Covered in both
tile forms: the tiny FP8 GEMM runs single-CTA tiles, the NVFP4 GEMM CTA
pairs (whose copies complete on the even CTA's barrier).  Run in a child
process (the binding loads one library per process, chosen by MOEQ_LIB)."""
import os
import subprocess
import sys

import pytest

from tests._util import need_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, time
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
from fp4_fp8_quantization_gb300 import moeq, synth
dev = "cuda"
ro = torch.from_numpy(np.array([0, 7, 23, 32], np.uint32).view(np.int32)).to(dev)
ids = torch.from_numpy(np.array([2, 0, 3], np.int32)).to(dev)
a = synth.e4m3_normal((32, 128), 1.0, seed=1, device=dev)
b = synth.e4m3_normal((4, 64, 128), 0.5, seed=2, device=dev)
sa = synth.uniform((32,), 0.01, 0.1, seed=3, device=dev)
sb = synth.uniform((4, 64), 0.005, 0.05, seed=4, device=dev)
c = torch.empty((32, 64), dtype=torch.bfloat16, device=dev)
moeq.clear_device_error()
t0 = time.time()
if sys.argv[2] == "fp8":
    moeq.grouped_matmul_rowwise_fp8(c, a, b, sa, sb, ro, ids, 16)
else:
    # NVFP4, 3 groups (300 / 1 / 140 rows), N = 512, K = 512: CTA-pair tiles
    K, N = 512, 512
    ro4 = np.array([0, 300, 301, 441], np.uint32)
    so4 = np.array([0, 384, 512, 768], np.uint32)
    ro = torch.from_numpy(ro4.view(np.int32)).to(dev)
    so = torch.from_numpy(so4.view(np.int32)).to(dev)
    a4 = synth.random_fp4_packed((441, K // 2), seed=5, device=dev)
    b4 = synth.random_fp4_packed((4, N, K // 2), seed=6, device=dev)
    asf = synth.random_bytes(moeq.sf_bytes(768, K // 16), 0x20, 0x30, seed=7, device=dev)
    bsf = synth.random_bytes(4 * moeq.sf_bytes(N, K // 16), 0x18, 0x28, seed=8, device=dev)
    es = synth.uniform((4,), 0.5, 2.0, seed=9, device=dev)
    c4 = torch.empty((441, N), dtype=torch.bfloat16, device=dev)
    moeq.grouped_matmul_blockscaled("nvfp4", c4, a4, asf, b4, bsf, es, ro, so, ids, N, K, 768)
torch.cuda.synchronize()
dt = time.time() - t0
bits = moeq.get_device_error()
moeq.clear_device_error()
after = moeq.get_device_error()
x = torch.arange(1 << 20, device=dev, dtype=torch.int64)
s = int(x.sum().item())
print("RESULT", bits, after, s == (1 << 20) * ((1 << 20) - 1) // 2, round(dt, 2))
"""


@pytest.mark.parametrize("form", ["fp8", "nvfp4_pair"])
def test_stuck_stage_times_out_and_context_survives(tmp_path, form):
    need_gpu()
    from fp4_fp8_quantization_gb300 import build
    lib = build.build(out_dir=str(tmp_path), defines=["MOEQ_TEST_STUCK_STAGE"])
    env = dict(os.environ, MOEQ_LIB=lib)
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, form], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT")][-1].split()
    bits, after, sum_ok, seconds = int(line[1]), int(line[2]), line[3] == "True", float(line[4])
    from fp4_fp8_quantization_gb300 import moeq
    assert bits & moeq.DEVERR_TIMEOUT          # the bounded wait ran out and said so
    assert after == 0                           # the bit clears
    assert sum_ok                               # the context still computes
    assert seconds < 30                         # every role left its wait
