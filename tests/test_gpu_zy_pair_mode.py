"""The tile form of the grouped GEMMs is a compile-time choice: CTA-pair
tiles (M=256 over two CTAs with tcgen05 cta_group::2, each CTA staging half
of the B tile) are the default for the FP4 kinds, single-CTA tiles for FP8
rowwise.  MOEQ_GEMM_PAIR=1 / =2 builds every kind in one form; this builds
both variants of the library and runs the GEMM and fused-SwiGLU parity tests
against each in a child process (the binding loads one library per process,
chosen by MOEQ_LIB), so the form the default build does not use for a kind
is covered too."""
import os
import subprocess
import sys

import pytest

from tests._util import need_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("pair", [1, 2])
def test_tile_form_build_passes_gemm_parity(tmp_path, pair):
    need_gpu()
    from fp4_fp8_quantization_gb300 import build
    lib = build.build(out_dir=str(tmp_path), defines=[f"MOEQ_GEMM_PAIR={pair}"])
    env = dict(os.environ, MOEQ_LIB=lib)
    sel = ("blockscaled_ragged_multitile or rowwise_fp8_ragged_multitile or "
           "rowwise_fp8_exact_invariants or fused_equals_chained_small or "
           "fused_mx_equals_chained")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_gemm.py", "tests/test_gpu_swiglu.py",
                        "tests/test_gpu_swiglu_mx.py", "-k", sel],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert " passed" in r.stdout
