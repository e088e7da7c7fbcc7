"""Grouped GEMMs, TEST INFRASTRUCTURE ONLY (see the package docstring).

Both GEMMs dequantize their operands to float64 and use one float64 matmul
per expert group; the result is rounded once to bf16.

* ``grouped_matmul_rowwise_fp8`` follows "grouped_matmul_rowwise_dynamic_scaled_fp8"
  (description and Args): for each token t of group g and channel n,
  out[t, n] = (sum_k a[t, k] * b[expert_ids[g], n, k]) * a_scale[t] * b_scale[expert_ids[g], n];
  ``b`` is [E, N, K] with K innermost; group g owns rows
  [a_offsets[g], a_offsets[g+1]).
* ``grouped_matmul_blockscaled`` follows "max.nn.moe.NvMxf4f8Strategy",
  ``grouped_matmul`` ("grouped NVIDIA block-scaled matmul with per-expert
  scales") and ``grouped_matmul_swiglu`` (``expert_scales``: per-expert
  matmul-epilogue scaling factors): out[t, n] = expert_scale[e] *
  sum_k (q_a[t,k] * sa[t, k/v]) * (q_b[e,n,k] * sb[e, n, k/v]).  The NVFP4
  weight's own tensor scale is taken to be folded into expert_scale; MX
  formats have no expert scale (1).
* Rows outside every group, and all rows of empty groups, are not written.
"""
import numpy as np

from . import formats as F
from . import layout as L


def _groups(a_offsets, expert_ids):
    for g in range(len(expert_ids)):
        r0, r1 = int(a_offsets[g]), int(a_offsets[g + 1])
        if r1 > r0:
            yield g, r0, r1, int(expert_ids[g])


def grouped_matmul_rowwise_fp8(a, b, a_scales, b_scales, a_offsets, expert_ids,
                               out=None, return_f64=False):
    """a: [T, K] E4M3 codes; b: [E, N, K] E4M3 codes; a_scales [T] fp32;
    b_scales [E, N] fp32.  Returns bf16 bits [T, N] (and optionally the
    float64 values before rounding, NaN where not written)."""
    a = np.asarray(a, np.uint8)
    b = np.asarray(b, np.uint8)
    T, K = a.shape
    E, N, Kb = b.shape
    assert Kb == K
    a_scales = np.asarray(a_scales, np.float32).reshape(-1).astype(np.float64)
    b_scales = np.asarray(b_scales, np.float32).reshape(E, N).astype(np.float64)
    out = np.zeros((T, N), np.uint16) if out is None else np.array(out, np.uint16)
    f64 = np.full((T, N), np.nan)
    for g, r0, r1, e in _groups(a_offsets, expert_ids):
        acc = F.decode_e4m3(a[r0:r1]) @ F.decode_e4m3(b[e]).T
        val = acc * a_scales[r0:r1, None] * b_scales[e][None, :]
        f64[r0:r1] = val
        out[r0:r1] = F.encode_bf16(val)
    return (out, f64) if return_f64 else out


def element_values(fmt, data, K):
    """Values of quantized elements: NVFP4 / MXFP4 packed E2M1 -> [.., K];
    MXFP8 E4M3 -> [.., K]."""
    data = np.asarray(data, np.uint8)
    if fmt in ("nvfp4", "mxfp4"):
        return F.decode_e2m1(F.unpack_e2m1(data))[..., :K]
    return F.decode_e4m3(data)[..., :K]


def scale_values(fmt, codes):
    return F.decode_e4m3(codes) if fmt == "nvfp4" else F.decode_e8m0(codes)


def weight_scales_logical(b_sf, E, N, kv):
    """Per-expert tiled weight scales -> [E, N, kv] logical bytes.  Each
    expert's block is the tiled layout of its [ceil128(N), kv] scales."""
    per = L.physical_bytes(N, kv)
    b_sf = np.asarray(b_sf, np.uint8).reshape(E, per)
    return np.stack([L.unswizzle(b_sf[e], N, kv) for e in range(E)])


def grouped_matmul_blockscaled(fmt, a, a_sf, b, b_sf, expert_scales, a_offsets,
                               a_scales_offsets, expert_ids, N, K,
                               scale_rows_total, out=None, return_f64=False,
                               row_scales=None):
    """a: [T, K/2] packed (NVFP4/MXFP4) or [T, K] (MXFP8); a_sf: flat tiled
    buffer of [scale_rows_total, K/v]; b: [E, N, K/2] or [E, N, K]; b_sf:
    per-expert tiled buffers.  Row t of group g uses scale row
    a_scales_offsets[g] + (t - a_offsets[g]).  row_scales (optional, [T]
    values of bf16 numbers): the per-row scale of grouped_matmul_swiglu,
    which the page applies together with the expert scale; multiplied in
    with the expert scale before the single rounding to bf16."""
    v = 16 if fmt == "nvfp4" else 32
    kv = K // v
    a = np.asarray(a, np.uint8)
    T = a.shape[0]
    b = np.asarray(b, np.uint8)
    E = b.shape[0]
    sa = scale_values(fmt, L.unswizzle(a_sf, scale_rows_total, kv))     # [rows, kv]
    sb = scale_values(fmt, weight_scales_logical(b_sf, E, N, kv))       # [E, N, kv]
    out = np.zeros((T, N), np.uint16) if out is None else np.array(out, np.uint16)
    f64 = np.full((T, N), np.nan)
    for g, r0, r1, e in _groups(a_offsets, expert_ids):
        p0 = int(a_scales_offsets[g])
        rg = r1 - r0
        deq_a = element_values(fmt, a[r0:r1], K) * np.repeat(sa[p0:p0 + rg], v, axis=1)
        deq_b = element_values(fmt, b[e], K) * np.repeat(sb[e], v, axis=1)
        acc = deq_a @ deq_b.T
        es = 1.0 if expert_scales is None else float(np.float32(expert_scales[e]))
        val = acc * es
        if row_scales is not None:
            val = val * np.asarray(row_scales, np.float64)[r0:r1, None]
        f64[r0:r1] = val
        out[r0:r1] = F.encode_bf16(val)
    return (out, f64) if return_f64 else out
