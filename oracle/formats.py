"""Element formats: E2M1 (fp4), E4M3 (fp8, the "fn" variant), E8M0, bf16.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages only name the formats: NVFP4 / MXFP4 / MXFP8 on
"grouped_quantize_dynamic_scaled_fp4_async_kernel" (description) and
"max.nn.moe.NvMxf4f8Strategy" (class description, ``is_nvfp4``); E8M0 for
MX scales on "Struct_ep_dispatch_mxfp4" (``execute``).  The definitions
below are the formats' own arithmetic definitions (OCP MX v1.0 element
formats; bf16 = the upper half of IEEE binary32), written out from those
definitions:

* decode: the value of each bit pattern, computed from sign / exponent /
  mantissa fields.
* encode: a *search over the code table* -- the finite code whose value is
  nearest to |x|, ties going to the even code (mantissa LSB 0); the sign of
  the result is the sign bit of x (so -0.0 and tiny negatives give a
  negative-zero code).  Searching only finite codes makes the encoders
  saturating ("satfinite"): anything beyond the largest finite magnitude
  encodes to it.
"""
import numpy as np

# ---------------------------------------------------------------- decoding


def e2m1_value(code):
    """Value of a 4-bit E2M1 code: sign bit 3, exponent bits 2..1 (bias 1),
    mantissa bit 0; exponent 0 is subnormal (0 or 0.5).  No inf / NaN."""
    code = int(code) & 0xF
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        mag = m * 0.5
    else:
        mag = 2.0 ** (e - 1) * (1.0 + m / 2.0)
    return s * mag


def e4m3_value(code):
    """Value of an 8-bit E4M3 ("fn") code: sign bit 7, exponent bits 6..3
    (bias 7), mantissa bits 2..0.  Exponent 0 is subnormal, 0x7F / 0xFF are
    NaN, there is no infinity; the largest finite magnitude is 448."""
    code = int(code) & 0xFF
    if code & 0x7F == 0x7F:
        return float("nan")
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0:
        mag = 2.0 ** -6 * (m / 8.0)
    else:
        mag = 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return s * mag


def e8m0_value(code):
    """Value of an 8-bit E8M0 scale code: 2**(code - 127); 255 is NaN."""
    code = int(code) & 0xFF
    if code == 0xFF:
        return float("nan")
    return 2.0 ** (code - 127)


def bf16_value(bits):
    """Value of a bf16 bit pattern: the upper 16 bits of an IEEE binary32."""
    b = np.array([int(bits) & 0xFFFF], dtype=np.uint32) << 16
    return float(b.view(np.float32)[0])


# Code tables (float64).  Index = code.
E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
E8M0_TABLE = np.array([e8m0_value(c) for c in range(256)], dtype=np.float64)

# Non-negative finite magnitudes in code order (code 0 .. max finite code);
# for these formats value increases with the code, which the searches use.
_E2M1_MAG = E2M1_TABLE[:8].copy()            # codes 0..7, 0 .. 6
_E4M3_MAG = E4M3_TABLE[:0x7F].copy()         # codes 0..126, 0 .. 448
assert np.all(np.diff(_E2M1_MAG) > 0) and np.all(np.diff(_E4M3_MAG) > 0)


def _bf16_mag_table():
    bits = np.arange(0, 0x7F81, dtype=np.uint32)      # 0 .. +inf
    return (bits << 16).view(np.float32).astype(np.float64)


_BF16_MAG = _bf16_mag_table()                 # codes 0x0000..0x7F80 (inf last)
assert np.all(np.diff(_BF16_MAG) > 0)


def decode_e2m1(codes):
    return E2M1_TABLE[np.asarray(codes, dtype=np.int64) & 0xF]


def decode_e4m3(codes):
    return E4M3_TABLE[np.asarray(codes, dtype=np.int64) & 0xFF]


def decode_e8m0(codes):
    return E8M0_TABLE[np.asarray(codes, dtype=np.int64) & 0xFF]


def decode_bf16(bits):
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32)


# ---------------------------------------------------------------- encoding


def _nearest_code(absx, mag):
    """Index of the entry of the increasing table ``mag`` nearest to each
    element of ``absx`` (>= 0), ties to the even index; beyond the last
    entry the last index (saturation)."""
    absx = np.asarray(absx, dtype=np.float64)
    n = mag.shape[0]
    hi = np.searchsorted(mag, absx, side="left")   # first entry >= absx
    hi = np.clip(hi, 0, n - 1)
    lo = np.clip(hi - 1, 0, n - 1)
    d_lo = absx - mag[lo]
    d_hi = mag[hi] - absx
    pick_hi = d_hi < d_lo
    tie = d_hi == d_lo
    even_hi = (hi & 1) == 0
    code = np.where(pick_hi | (tie & even_hi), hi, lo)
    code = np.where(absx >= mag[n - 1], n - 1, code)  # saturate
    return code.astype(np.int64)


def encode_e2m1(x):
    """Nearest E2M1 code (ties to even code, satfinite, sign kept)."""
    x = np.asarray(x, dtype=np.float64)
    mag = _nearest_code(np.abs(x), _E2M1_MAG)
    return (mag | (np.signbit(x).astype(np.int64) << 3)).astype(np.uint8)


def encode_e4m3(x):
    """Nearest finite E4M3 code (ties to even code, satfinite, sign kept)."""
    x = np.asarray(x, dtype=np.float64)
    mag = _nearest_code(np.abs(x), _E4M3_MAG)
    return (mag | (np.signbit(x).astype(np.int64) << 7)).astype(np.uint8)


def encode_bf16(x):
    """bf16 bit pattern nearest to x (round to nearest, ties to even);
    magnitudes at or above the midpoint between the largest finite bf16 and
    2**128 become infinity, as IEEE rounding does."""
    x = np.asarray(x, dtype=np.float64)
    finite = _BF16_MAG[:-1]
    mag = _nearest_code(np.abs(x), finite)
    overflow_at = finite[-1] + (2.0 ** 128 - finite[-1]) / 2.0
    mag = np.where(np.abs(x) >= overflow_at, 0x7F80, mag)
    return (mag | (np.signbit(x).astype(np.int64) << 15)).astype(np.uint16)


def round_bf16(x):
    """x rounded to the nearest bf16 value, returned as float32."""
    return decode_bf16(encode_bf16(x))


# ---------------------------------------------------------------- packing


def pack_e2m1(codes):
    """Two E2M1 codes per byte along the last axis; the element with the
    lower index goes to the low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    assert codes.shape[-1] % 2 == 0
    lo = codes[..., 0::2] & 0xF
    hi = codes[..., 1::2] & 0xF
    return (lo | (hi << 4)).astype(np.uint8)


def unpack_e2m1(packed):
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out
