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
* silu(g) = g / (1 + exp_spec(-g)) in float32, where ``exp_spec`` is this
  project's own exponential: Cody-Waite argument reduction (W. J. Cody and
  W. Waite, "Software Manual for the Elementary Functions", 1980) with ln 2
  split into a 16-significant-bit head and a tail, then the degree-7 Taylor
  polynomial of e^f evaluated by Horner's rule with separately rounded fp32
  multiplies and adds, then scaling by 2^n through two exact power-of-two
  multiplies.  The same steps run in the CUDA kernels, so both sides produce
  the same bits; its accuracy is checked against long-double exp.
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
EXP_OVERFLOW_X = F32(89.0)      # e^89 > largest fp32: +inf
EXP_UNDERFLOW_X = F32(-104.0)   # e^-104 < half the smallest fp32 subnormal: 0


def exp_spec(x):
    """float32 exponential, defined step by step (see the module docstring)."""
    x = np.asarray(x, dtype=F32)
    with np.errstate(over="ignore", under="ignore", invalid="ignore"):
        xc = np.clip(x, EXP_UNDERFLOW_X, EXP_OVERFLOW_X).astype(F32)
        n = np.rint(xc * LOG2E).astype(F32)              # round half even
        f = (xc - n * LN2_HI).astype(F32)
        f = (f - n * LN2_LO).astype(F32)
        p = EXP_COEF[7]
        for k in range(6, -1, -1):
            p = (p * f).astype(F32)
            p = (p + EXP_COEF[k]).astype(F32)
        ni = n.astype(np.int64)
        n1 = ni >> 1                                   # floor(n / 2)
        n2 = ni - n1
        s1 = np.ldexp(F32(1.0), n1).astype(F32)
        s2 = np.ldexp(F32(1.0), n2).astype(F32)
        r = ((p * s1).astype(F32) * s2).astype(F32)
    r = np.where(x >= EXP_OVERFLOW_X, F32(np.inf), r)
    r = np.where(x <= EXP_UNDERFLOW_X, F32(0.0), r)
    return r.astype(F32)


def silu_spec(g):
    """silu(g) = g / (1 + exp_spec(-g)), each step one fp32 operation."""
    g = np.asarray(g, dtype=F32)
    d = (F32(1.0) + exp_spec(-g)).astype(F32)
    with np.errstate(divide="ignore", invalid="ignore"):
        return (g / d).astype(F32)


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
