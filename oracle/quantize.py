"""Block quantizers and the grouped (ragged, per-expert padded) quantizer.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources.
* "grouped_quantize_dynamic_scaled_fp4_async_kernel" (description): each
  block of work finds its expert from ``row_offsets`` / ``scales_offsets`` and
  quantizes that expert's BF16 rows to NVFP4 / MXFP4 / MXFP8, writing block
  scale factors; ``sf_tensor`` is a read-only per-expert fp32 tensor-wise
  scale.
* "max.nn.moe.NvMxf4f8Strategy", ``grouped_quantize``: per-expert
  quantization with the scales padded per expert.
* The pages fix no formula.  The readings used here (stated once, used by
  the oracle and the kernels alike):
  - NVFP4: 16-element blocks, E2M1 elements, E4M3 block scale, per-expert
    fp32 tensor scale s_e = amax_e / (6 * 448) (``tensor_scale_from_amax``),
    and the fixed fp32 operation order of ``nvfp4_quantize_blocks``.
  - MXFP8 / MXFP4: 32-element blocks, E8M0 scale chosen by the OCP MX v1.0
    floor rule (``mx_quantize_blocks``).
  - Padded scale rows: expert group g owns logical scale rows
    [scales_offsets[g], scales_offsets[g+1]); its r_g data rows come first,
    then the rows up to the next multiple of 128 (ceil(r_g / 128) * 128 rows
    in all) are written as zero bytes.  Any further rows of the range, and
    rows at or beyond scales_offsets[G], are not touched.

All float32 steps are numpy float32 operations: one IEEE binary32 operation
each, round-to-nearest-even, no fused multiply-add.
"""
import numpy as np

from . import formats as F
from . import layout as L

F32 = np.float32
NVFP4_BLOCK = 16
MX_BLOCK = 32
# 6 = largest E2M1 magnitude, 448 = largest E4M3 magnitude.
NVFP4_TENSOR_DIVISOR = F32(6.0 * 448.0)


def block_size(fmt):
    return NVFP4_BLOCK if fmt == "nvfp4" else MX_BLOCK


def tensor_scale_from_amax(amax):
    """Per-expert NVFP4 tensor scale (dequantization direction):
    s = fp32(amax / 2688); an all-zero (or empty) expert gets s = 1."""
    amax = np.asarray(amax, dtype=F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        s = amax / NVFP4_TENSOR_DIVISOR
    return np.where(amax == F32(0), F32(1), s).astype(F32)


def group_amax(x, row_offsets, expert_ids, num_experts):
    """amax_e = max |x| over every row of every group routed to expert e
    (0 for experts with no rows).  Exact (max of magnitudes)."""
    x = np.asarray(x, dtype=F32)
    amax = np.zeros(num_experts, dtype=F32)
    for g in range(len(expert_ids)):
        r0, r1 = int(row_offsets[g]), int(row_offsets[g + 1])
        if r1 > r0:
            e = int(expert_ids[g])
            amax[e] = max(amax[e], np.abs(x[r0:r1]).max())
    return amax


def nvfp4_quantize_blocks(x, s):
    """NVFP4 quantization of 16-element blocks.

    x: [..., 16] float32 values; s: float32 tensor scale broadcastable to
    x[..., 0].  Steps (each one fp32 operation):
      1. inv = 1 / s
      2. m = max |x_i| over the block
      3. sb_f = (m * inv) / 6 ; sb_code = E4M3(sb_f) ; sb = value(sb_code)
      4. sb == 0: every element code is +0; else r = inv / sb and
         q_i = E2M1(x_i * r)
    Dequantized value: value(q_i) * sb * s.
    Returns (element codes [..., 16] uint8, scale codes [...] uint8).
    """
    x = np.asarray(x, dtype=F32)
    assert x.shape[-1] == NVFP4_BLOCK
    s = np.asarray(s, dtype=F32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        inv = F32(1.0) / s
        m = np.abs(x).max(axis=-1)
        sb_f = (m * inv) / F32(6.0)
        sb_code = F.encode_e4m3(sb_f)
        sb = F.decode_e4m3(sb_code).astype(F32)
        r = inv / sb
        v = x * np.asarray(r, dtype=F32)[..., None]
    q = F.encode_e2m1(v)
    q = np.where((sb == F32(0))[..., None], np.uint8(0), q).astype(np.uint8)
    return q, sb_code.astype(np.uint8)


def mx_quantize_blocks(x, elem):
    """MX quantization of 32-element blocks (OCP MX v1.0 floor rule).

    elem: "e4m3" (MXFP8, largest element exponent emax = 8) or "e2m1"
    (MXFP4, emax = 2).
      1. m = max |x_i|
      2. m == 0: scale code 0 and every element code is +0
      3. E = floor(log2 m) (exact); c = clamp(E - emax + 127, 0, 254)
      4. q_i = elem(x_i * 2**(127 - c)), the product exact in float64,
         saturating at the element format's largest magnitude.
    Returns (element codes [..., 32] uint8, scale codes [...] uint8).
    """
    x = np.asarray(x, dtype=np.float64)
    assert x.shape[-1] == MX_BLOCK
    emax = 8 if elem == "e4m3" else 2
    m = np.abs(x).max(axis=-1)
    zero = m == 0
    _, ex = np.frexp(np.where(zero, 1.0, m))        # m = f * 2**ex, f in [0.5, 1)
    E = ex.astype(np.int64) - 1
    c = np.clip(E - emax + 127, 0, 254)
    c = np.where(zero, 0, c)
    v = x * np.ldexp(1.0, (127 - c))[..., None]
    enc = F.encode_e4m3 if elem == "e4m3" else F.encode_e2m1
    q = enc(v)
    q = np.where(zero[..., None], np.uint8(0), q).astype(np.uint8)
    return q, c.astype(np.uint8)


def quantize_rows(fmt, x, s=None):
    """Quantize [R, K] rows.  Returns (element bytes, logical scales [R, K/v]).
    Element bytes: NVFP4 / MXFP4 packed two per byte [R, K/2]; MXFP8 [R, K]."""
    x = np.asarray(x, dtype=F32)
    R, K = x.shape
    v = block_size(fmt)
    assert K % v == 0
    blocks = x.reshape(R, K // v, v)
    if fmt == "nvfp4":
        q, sc = nvfp4_quantize_blocks(blocks, np.broadcast_to(np.asarray(s, F32), (R, 1)))
    elif fmt == "mxfp8":
        q, sc = mx_quantize_blocks(blocks, "e4m3")
    elif fmt == "mxfp4":
        q, sc = mx_quantize_blocks(blocks, "e2m1")
    else:
        raise ValueError(fmt)
    q = q.reshape(R, K)
    if fmt in ("nvfp4", "mxfp4"):
        q = F.pack_e2m1(q)
    return q, sc.reshape(R, K // v)


def grouped_quantize(fmt, x, row_offsets, scales_offsets, expert_ids,
                     tensor_scale=None, out=None, scales=None,
                     scale_rows_total=None):
    """The grouped quantizer.

    x: [T, K] float32 (BF16 values for activations).  Group g owns input
    rows [row_offsets[g], row_offsets[g+1]) and logical scale rows
    [scales_offsets[g], scales_offsets[g+1]); NVFP4 uses the tensor scale
    tensor_scale[expert_ids[g]].  ``out`` / ``scales`` are the initial
    buffers (their other bytes are returned unchanged); the scale buffer is
    the flat tiled layout of ``layout`` with scale_rows_total logical rows.
    """
    x = np.asarray(x, dtype=F32)
    T, K = x.shape
    v = block_size(fmt)
    kv = K // v
    ob = K if fmt == "mxfp8" else K // 2
    if scale_rows_total is None:
        scale_rows_total = int(scales_offsets[-1])
    out = np.zeros((T, ob), np.uint8) if out is None else np.array(out, dtype=np.uint8)
    nbytes = L.physical_bytes(scale_rows_total, kv)
    scales = np.zeros(nbytes, np.uint8) if scales is None else np.array(scales, dtype=np.uint8).reshape(-1)
    for g in range(len(expert_ids)):
        r0, r1 = int(row_offsets[g]), int(row_offsets[g + 1])
        p0, p1 = int(scales_offsets[g]), int(scales_offsets[g + 1])
        rg = r1 - r0
        assert rg >= 0 and p1 - p0 >= rg and p0 % 128 == 0
        padded = (rg + 127) // 128 * 128
        logical = np.zeros((padded, kv), np.uint8)
        if rg > 0:
            s = None
            if fmt == "nvfp4":
                s = F32(tensor_scale[int(expert_ids[g])])
            q, sc = quantize_rows(fmt, x[r0:r1], s)
            out[r0:r1] = q
            logical[:rg] = sc
        rr, cc = np.meshgrid(np.arange(p0, p0 + padded), np.arange(kv), indexing="ij")
        scales[L.sf_offset(rr, cc, kv)] = logical
    return out, scales


def gather_rows(x, indices, divisor):
    """The rows the gather-fused quantizer works on ("max.nn.moe.NvMxf4f8Strategy",
    grouped_quantize: indices, indices_divisor).  Reading adopted: row t of
    the quantized matrix is input row indices[t] // divisor."""
    idx = np.asarray(indices, dtype=np.int64)
    assert divisor >= 1 and np.all(idx >= 0)
    return np.asarray(x)[idx // int(divisor)]


def padded_scale_offsets(row_offsets):
    """scales_offsets[g] = sum over h < g of ceil(r_h / 128) * 128."""
    ro = np.asarray(row_offsets, dtype=np.int64)
    r = np.diff(ro)
    pad = (r + 127) // 128 * 128
    return np.concatenate([[0], np.cumsum(pad)]).astype(np.uint32)
