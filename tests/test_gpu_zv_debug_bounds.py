"""Debug-bounds build: with MOEQ_DEBUG_BOUNDS every global store of the
kernels is checked against its buffer's extent (a store outside it would be
skipped and flagged with MOEQ_DEVERR_BOUNDS).  This builds that variant and
runs the quantizer, GEMM, SwiGLU and layout parity tests against it in a
child process, where a fixture asserts after every test that no store was
flagged (the binding loads one library per process, chosen by MOEQ_LIB)."""
import os
import subprocess
import sys

import pytest

from tests._util import need_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_debug_bounds_build_flags_no_store(tmp_path):
    need_gpu()
    from fp4_fp8_quantization_gb300 import build
    lib = build.build(out_dir=str(tmp_path), defines=["MOEQ_DEBUG_BOUNDS"])
    env = dict(os.environ, MOEQ_LIB=lib, MOEQ_CHECK_BOUNDS="1")
    sel = ("ragged or special or strided or gather or multitile or tiny or "
           "fused_equals_chained_small or fused_mx_equals_chained or bit_exact or sf_swizzle")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_quantize.py", "tests/test_gpu_gemm.py",
                        "tests/test_gpu_swiglu.py", "tests/test_gpu_swiglu_mx.py",
                        "tests/test_gpu_layout.py", "-k", sel],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
