"""The C ABI without a GPU: the library loads, exports every function that
include/moeq.h declares, and rejects bad host arguments before launching
anything (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from fp4_fp8_quantization_gb300 import moeq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "moeq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moeq_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(moeq._LIB_PATH):
        from fp4_fp8_quantization_gb300 import build
        build.build()
    return moeq.lib()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(moeq.EXPORTS)


def test_status_strings(lib):
    for code, name in moeq.STATUS.items():
        assert lib.moeq_status_string(code).decode() == name


P = ctypes.c_void_p
FAKE = P(0x10000)          # 16-byte aligned, never dereferenced
ODD = P(0x10004)


def test_quantize_rejects_bad_host_arguments(lib):
    f = lib.moeq_grouped_quantize
    ok = dict(fmt=0, inp=FAKE, stride=256, rows=10, K=256, out=FAKE, sf=FAKE, srows=128,
              ro=FAKE, so=FAKE, ids=FAKE, ts=FAKE, E=4, mt=10, G=2, s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["fmt"], a["inp"], a["stride"], a["rows"], a["K"], a["out"], a["sf"],
                 a["srows"], a["ro"], a["so"], a["ids"], a["ts"], a["E"], a["mt"], a["G"], a["s"])

    assert call(K=100) == 1                # K % 128
    assert call(stride=200) == 1           # stride < K
    assert call(srows=100) == 1            # scale rows % 128
    assert call(ts=None) == 1              # NVFP4 without tensor scale (ValueError analogue)
    assert call(fmt=7) == 1
    assert call(ro=None) == 1
    assert call(E=0) == 1
    assert call(G=-1) == 1
    assert call(inp=ODD) == 1              # misaligned
    assert call(G=0) == 0                  # no groups: OK, nothing launched
    assert call(fmt=2, ts=None, G=0) == 0  # MX needs no tensor scale


def test_layout_helpers_reject_bad_host_arguments(lib):
    sw, un, il = lib.moeq_sf_swizzle, lib.moeq_sf_unswizzle, lib.moeq_interleave_gate_up
    for f in (sw, un):
        assert f(FAKE, FAKE, -1, 128, 4, None) == 1    # negative sizes
        assert f(FAKE, FAKE, 1, -5, 4, None) == 1
        assert f(None, FAKE, 1, 128, 4, None) == 1     # NULL with work to do
        assert f(FAKE, None, 1, 128, 4, None) == 1
        assert f(None, None, 0, 128, 4, None) == 0     # empty: OK, nothing launched
        assert f(None, None, 3, 0, 4, None) == 0
        assert f(FAKE, FAKE, 1 << 41, 128, 4, None) == 1   # beyond the size limit
    assert il(FAKE, FAKE, FAKE, 1, -1, 16, None) == 1
    assert il(FAKE, None, FAKE, 1, 4, 16, None) == 1
    assert il(None, None, None, 2, 4, 0, None) == 0


def test_route_and_dispatch_reject_bad_host_arguments(lib):
    r = lib.moeq_route_topk

    def route(ids=FAKE, T=8, k=2, E=4, ro=FAKE, eids=FAKE, src=FAKE, dst=None, so=FAKE, slot=0):
        return r(ids, T, k, E, ro, eids, src, dst, so, slot, None)

    assert route(k=0) == 1                  # top_k < 1
    assert route(E=0) == 1                  # no experts
    assert route(E=2000) == 2               # above 1024 experts
    assert route(slot=100) == 1             # slot % 128
    assert route(ro=None) == 1              # row_offsets
    assert route(ids=None) == 1             # topk_ids with tokens
    assert route(src=ODD) == 1              # misaligned
    assert route(dst=ODD) == 1
    assert route(T=1 << 30, k=4) == 2       # 2^32 choices
    rows = lib.moeq_dispatch_scale_rows
    rows.restype = ctypes.c_int64
    assert rows(100, 8, 16, 0) == (800 + 127 * 16) // 128 * 128
    assert rows(100, 8, 16, 256) == 16 * 256
    assert rows(-1, 8, 16, 0) == -1
    d = lib.moeq_dispatch_mxfp4
    ok = dict(tok=FAKE, stride=256, T=8, H=256, ids=FAKE, k=2, E=4, out=FAKE, sf=FAKE,
              srows=rows(8, 2, 4, 0), ro=FAKE, eids=FAKE, src=FAKE, dst=FAKE, so=FAKE, slot=0,
              s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return d(a["tok"], a["stride"], a["T"], a["H"], a["ids"], a["k"], a["E"], a["out"],
                 a["sf"], a["srows"], a["ro"], a["eids"], a["src"], a["dst"], a["so"], a["slot"],
                 a["s"])

    assert call(H=200) == 1                 # hidden % 128
    assert call(stride=128) == 1            # stride < hidden
    assert call(srows=0) == 1               # no scale rows
    assert call(srows=ok["srows"] - 128) == 1   # fewer scale rows than needed
    assert call(so=None) == 1               # scale offsets required
    assert call(dst=None) == 1              # the inverse map is required
    assert call(out=ODD) == 1
    assert call(slot=128, srows=4 * 128 - 128) == 1
    assert call(k=9, srows=rows(8, 9, 4, 0)) == 2   # token-major quantization: top_k <= 8
    q = lib.moeq_quantize_topk
    okq = dict(fmt=0, tok=FAKE, stride=256, T=8, K=256, ids=FAKE, k=2, dst=FAKE, ro=FAKE,
               so=FAKE, ts=FAKE, E=4, out=FAKE, sf=FAKE, srows=512, s=None)

    def callq(**kw):
        a = dict(okq, **kw)
        return q(a["fmt"], a["tok"], a["stride"], a["T"], a["K"], a["ids"], a["k"], a["dst"],
                 a["ro"], a["so"], a["ts"], a["E"], a["out"], a["sf"], a["srows"], a["s"])

    assert callq(fmt=5) == 1
    assert callq(K=100) == 1                # K % 128
    assert callq(ts=None) == 1              # NVFP4 needs the tensor scales
    assert callq(dst=None) == 1
    assert callq(srows=100) == 1
    assert callq(k=9) == 2                  # top_k <= 8


def test_gemms_reject_bad_host_arguments(lib):
    r = lib.moeq_grouped_matmul_rowwise_fp8
    #        c     a     b     sa    sb    ao    ids   T   N    K    E  mt  G  stream
    assert r(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 64, 100, 2, 8, 2, None) == 1  # K
    assert r(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 72, 128, 2, 8, 2, None) == 1  # N % 16
    assert r(FAKE, FAKE, None, FAKE, FAKE, FAKE, FAKE, 64, 64, 128, 2, 8, 2, None) == 1  # b
    assert r(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 64, 128, 2, 8, 2000, None) == 2
    assert r(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 64, 128, 2, 8, 0, None) == 0
    bs = lib.moeq_grouped_matmul_blockscaled
    args = [0] + [FAKE] * 9 + [64, 128, 128, 512, 2, 8, 2, None]
    a = list(args); a[0] = 1; a[13] = 384                    # MXFP4 needs K % 256
    assert bs(*a) == 1
    a = list(args); a[0] = 7                                 # unknown format
    assert bs(*a) == 1
    a = list(args); a[0] = 0; a[6] = None                    # NVFP4 without expert scales
    assert bs(*a) == 1
    a = list(args); a[0] = 0; a[13] = 384                    # NVFP4 needs K % 256
    assert bs(*a) == 1
    a = list(args); a[0] = 2; a[6] = None; a[12] = 192       # N % 128
    assert bs(*a) == 1
    sw = lib.moeq_grouped_matmul_swiglu
    sargs = [FAKE] * 12 + [64, 128, 64, 512, 2, 8, 2, None]
    a = list(sargs); a[7] = None                             # missing SiLU-output scale
    assert sw(*a) == 1
    a = list(sargs); a[14] = 96                              # I % 64
    assert sw(*a) == 1
    a = list(sargs); a[8] = ODD                              # unaligned row scales
    assert sw(*a) == 1
    mx = lib.moeq_grouped_matmul_swiglu_mx
    margs = [1] + [FAKE] * 10 + [64, 128, 128, 512, 2, 8, 2, None]
    a = list(margs); a[0] = 0                                # NVFP4 is not an MX format
    assert mx(*a) == 1
    a = list(margs); a[13] = 64                              # I % 128
    assert mx(*a) == 1
    a = list(margs); a[0] = 1; a[14] = 384                   # MXFP4 needs K % 256
    assert mx(*a) == 1
    a = list(args); a[0] = 0; a[16] = 1025                  # more groups than the scheduler
    assert bs(*a) == 2
    qm = lib.moeq_swiglu_quantize_mx
    assert qm(0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 128, 128, 2, 8, 2, None) == 1
    assert qm(2, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 128, 64, 2, 8, 2, None) == 1
    q = lib.moeq_swiglu_quantize
    assert q(FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 64, 128, 64, 2, 8, 2, None) == 1
    assert q(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 64, 128, 48, 2, 8, 2, None) == 1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(moeq, "_lib", None)
    monkeypatch.setattr(moeq, "_LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        moeq.lib()
