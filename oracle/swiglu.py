"""SiLU definition and the chained SwiGLU + NVFP4 requantization.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Sources: "max.nn.moe.NvMxf4f8Strategy" -- ``fused_silu_quantize`` applies the
gated activation and then quantizes; ``grouped_matmul_swiglu`` is the same
computation fused into one kernel, whose (packed, scales) output matches the
chained path byte for byte with a bf16 rounding where the chained path has a
bf16 tensor (``match_bf16``); ``input_scales`` is the raw per-expert SiLU
output scale and the quantizer consumes its inverse
(``prepare_swiglu_operands``).

Readings (the pages give no formulas):
* gate/up arrangement: in the [T, 2I] GEMM output, column 2j is gate_j and
  column 2j+1 is up_j (granularity-1 interleave).
* h_j = silu(gate_j) * up_j in float32, not rounded to bf16, then NVFP4
  quantized with the expert's raw output scale s_e (inverted inside).
* silu(g) = g * sigma(g) in float32, where sigma is this project's own
  logistic function, every step one IEEE fp32 operation (round to nearest
  even) or one fused multiply-add (a single rounding):
    e     = exp_neg_spec(-|g|)            (e in [0, 1])
    d     = 1 + e                         (d in [1, 2])
    r     = recip_spec(d)                 (1 / d)
    sigma = r if g >= 0 else e * r        (e / (1 + e) = 1 / (1 + e^-g))
  ``exp_neg_spec`` is Cody-Waite argument reduction (W. J. Cody and
  W. Waite, "Software Manual for the Elementary Functions", 1980) with ln 2
  split into a 16-significant-bit head and a tail, the degree-7 Taylor
  polynomial of e^f by Horner's rule in fused multiply-adds, and a scaling by
  2^n (taken as 0 below the smallest normal power, n < -126).
  ``recip_spec`` is Newton-Raphson reciprocal iteration from the linear
  seed 24/17 - 8/17 d, three steps.  The same steps run in the CUDA
  kernels, so both sides produce the same bits; the accuracy is checked
  against long-double exp and float64 SiLU.  The fp32 fused multiply-add is
  emulated exactly in ``fma_f32``.
"""
import math

import numpy as np

from . import quantize as Q

F32 = np.float32

# ln 2 rounded to 16 significant bits (45426 / 65536), so that n * LN2_HI is
# exact for |n| < 2**8; the tail is the fp32 rounding of the remainder.
LN2_HI = F32(45426.0 / 65536.0)
LN2_LO = F32(math.log(2.0) - 45426.0 / 65536.0)
LOG2E = F32(1.0 / math.log(2.0))
# Taylor coefficients 1/k!, k = 0..7, rounded to fp32.
EXP_COEF = [F32(1.0 / math.factorial(k)) for k in range(8)]
EXP_ARG_MIN = F32(-104.0)       # arguments below are clamped (e^-104 = 0 here)
# 1.5 * 2^23: adding it rounds a value of magnitude < 2^22 to an integer
# (ties to even); subtracting it again is exact.
ROUND_SHIFT = F32(12582912.0)
# linear seed of the reciprocal on [1, 2]: 24/17 - 8/17 d (the minimax line:
# relative error at most 1/17, reached at d = 1, 3/2 and 2), constants
# rounded to fp32
RECIP_SEED_A = F32(24.0 / 17.0)
RECIP_SEED_B = F32(8.0 / 17.0)
RECIP_STEPS = 3


def fma_f32(a, b, c):
    """fp32 fused multiply-add: a * b + c rounded once to nearest even.

    a * b of two fp32 numbers is exact in float64 (48 significant bits).  The
    float64 sum is rounded to odd (round to nearest, then, if inexact and the
    last significand bit is even, step to the neighbour on the side of the
    exact value; the error comes from Knuth's TwoSum), and a round-to-odd
    result in 53 bits rounds to the correct nearest-even fp32 value
    (S. Boldo and G. Melquiond, "Emulation of FMA and correctly rounded sums:
    proved algorithms using rounding to odd", IEEE Trans. Computers, 2008).
    """
    a, b, c = np.broadcast_arrays(np.asarray(a, F32), np.asarray(b, F32),
                                  np.asarray(c, F32))
    p = a.astype(np.float64) * b.astype(np.float64)          # exact
    c64 = c.astype(np.float64)
    with np.errstate(invalid="ignore", over="ignore"):
        s = p + c64
        bv = s - p
        err = (p - (s - bv)) + (c64 - bv)                     # exact error
        even = (np.asarray(s, np.float64).view(np.int64) & 1) == 0
        fix = np.isfinite(s) & (err != 0) & even
        s = np.where(fix, np.nextafter(s, np.where(err > 0, np.inf, -np.inf)), s)
        return s.astype(F32)


def exp_neg_spec(x):
    """e^x for x <= 0 (or NaN, which gives 0), defined step by step:
    x clamped to >= -104; n = nearest integer to x * log2(e) (one fused
    multiply-add with the 1.5 * 2^23 shift, then the shift taken off);
    f = x - n ln2 in two fused multiply-adds (head, tail); p = Horner of the
    degree-7 Taylor polynomial in fused multiply-adds; result p * 2^n, with
    2^n taken as 0 for n < -126."""
    x = np.asarray(x, dtype=F32)
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        xc = np.fmax(x, EXP_ARG_MIN).astype(F32)             # NaN -> -104
        t = fma_f32(xc, LOG2E, ROUND_SHIFT)
        n = (t - ROUND_SHIFT).astype(F32)
        f = fma_f32(-n, LN2_HI, xc)
        f = fma_f32(-n, LN2_LO, f)
        p = np.full(x.shape, EXP_COEF[7], F32)
        for k in range(6, -1, -1):
            p = fma_f32(p, f, EXP_COEF[k])
        ni = n.astype(np.int64)
        s = np.where(ni >= -126, np.ldexp(1.0, np.maximum(ni, -126)), 0.0).astype(F32)
        return (p * s).astype(F32)


def recip_spec(d):
    """1 / d for d in [1, 2]: r0 = 24/17 - 8/17 d (one fused multiply-add),
    then three Newton-Raphson steps q = 1 - d r, r = r + r q (each a fused
    multiply-add)."""
    d = np.asarray(d, dtype=F32)
    r = fma_f32(d, -RECIP_SEED_B, RECIP_SEED_A)
    for _ in range(RECIP_STEPS):
        q = fma_f32(-d, r, F32(1.0))
        r = fma_f32(r, q, r)
    return r


def sigmoid_spec(g):
    """sigma(g) = 1 / (1 + e^-g) through e = e^-|g| (see the module
    docstring)."""
    g = np.asarray(g, dtype=F32)
    e = exp_neg_spec(-np.abs(g))
    r = recip_spec((F32(1.0) + e).astype(F32))
    with np.errstate(invalid="ignore"):
        return np.where(g >= 0, r, (e * r).astype(F32)).astype(F32)


def silu_spec(g):
    """silu(g) = g * sigma(g), one fp32 multiply."""
    g = np.asarray(g, dtype=F32)
    with np.errstate(invalid="ignore", under="ignore"):
        return (g * sigmoid_spec(g)).astype(F32)


def swiglu(y):
    """y: [.., 2I] float32 (bf16 values), gate/up interleaved -> h [.., I]."""
    y = np.asarray(y, dtype=F32)
    g = y[..., 0::2]
    u = y[..., 1::2]
    return (silu_spec(g) * u).astype(F32)


def swiglu_quantize(y, out_tensor_scale, a_offsets, a_scales_offsets,
                    expert_ids, out=None, scales=None, scale_rows_total=None,
                    fmt="nvfp4"):
    """Chained SwiGLU + quantization of the bf16 GEMM output y [T, 2I].

    fmt "nvfp4": with the raw per-expert output scale s_e =
    out_tensor_scale[e]; output packed [T, I/2] and the tiled scale buffer of
    [rows, I/16].  fmt "mxfp4" / "mxfp8" (the strategy's MX formats, no
    tensor scale): the MX block rule on the fp32 h values; output [T, I/2]
    packed E2M1 or [T, I] E4M3 and E8M0 scales of [rows, I/32].  Scale rows
    are padded per expert as for the activations."""
    h = swiglu(y)
    return Q.grouped_quantize(fmt, h, a_offsets, a_scales_offsets, expert_ids,
                              tensor_scale=out_tensor_scale if fmt == "nvfp4" else None,
                              out=out, scales=scales,
                              scale_rows_total=scale_rows_total)
