"""Builds libmoeq.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel, then linked into one
shared library (CUDA runtime linked statically, so the library loads on a
machine without a GPU driver).  Run as ``python -m fp4_fp8_quantization_gb300.build``.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoeq.so")
SOURCES = ["api.cu", "quantize.cu", "gemm.cu", "layout.cu", "route.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC",
         "-I" + os.path.join(ROOT, "include")]


def _compile(src, verbose, build_dir, extra):
    obj = os.path.join(build_dir, src.replace(".cu", ".o"))
    cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r


def build(verbose=False, out_dir=None, defines=()):
    """Builds libmoeq.so in the package, or, with out_dir, a variant of it
    in out_dir compiled with extra preprocessor definitions (defines, e.g.
    ["MOEQ_GEMM_PAIR=2"]) and returns its path."""
    build_dir = BUILD if out_dir is None else os.path.join(out_dir, "_build")
    lib_path = LIB if out_dir is None else os.path.join(out_dir, "libmoeq.so")
    extra = ["-D" + d for d in defines]
    os.makedirs(build_dir, exist_ok=True)
    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose, build_dir, extra), SOURCES))
    failed = False
    for src, _, r in results:
        if r.returncode != 0 or verbose:
            sys.stderr.write(f"--- {src}\n{r.stdout}{r.stderr}")
        failed |= r.returncode != 0
    if failed:
        raise RuntimeError("nvcc failed")
    objs = [o for _, o, _ in results]
    tmp = lib_path + ".tmp"
    r = subprocess.run([NVCC, *ARCH, "-shared", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
