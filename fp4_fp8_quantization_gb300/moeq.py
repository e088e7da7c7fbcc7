"""Python binding of the moeq C ABI (``include/moeq.h``).

Argument marshalling only: each function checks that the tensors it is given
are CUDA tensors of the documented dtype and layout, passes their device
pointers and sizes to the function of the same name in ``libmoeq.so`` on the
current CUDA stream (or ``stream``), and raises ``MoeqError`` on a non-OK
status.  Every step of the computation runs in the library's CUDA kernels;
there is no other implementation, and importing a function whose library is
missing raises.
"""
import ctypes
import os

import torch

# The in-tree library, or another build of it named by MOEQ_LIB (e.g. one
# compiled with different tile options by build.build(variant_dir, flags)).
_LIB_PATH = os.environ.get("MOEQ_LIB") or os.path.join(
    os.path.dirname(os.path.abspath(__file__)), "libmoeq.so")
_lib = None

FORMATS = {"nvfp4": 0, "mxfp4": 1, "mxfp8": 2}
STATUS = {0: "MOEQ_OK", 1: "MOEQ_ERR_INVALID_ARG", 2: "MOEQ_ERR_UNSUPPORTED",
          3: "MOEQ_ERR_CUDA", 4: "MOEQ_ERR_DEVICE"}
DEVERR_BAD_OFFSETS, DEVERR_BAD_EXPERT, DEVERR_SCALE_ROWS, DEVERR_TIMEOUT, DEVERR_BAD_INDEX = 1, 2, 4, 8, 16
DEVERR_BOUNDS = 32   # debug builds only: a store outside its buffer was skipped

_P, _I64, _I32, _U32P = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.POINTER(ctypes.c_uint32)
_SIGNATURES = {
    "moeq_grouped_amax_scale": [_P, _I64, _I64, _I64, _P, _P, _P, _I32, _I32, _P],
    "moeq_grouped_quantize": [_I32, _P, _I64, _I64, _I64, _P, _P, _I64, _P, _P, _P, _P,
                              _I32, _I32, _I32, _P],
    "moeq_grouped_amax_scale_gather": [_P, _I64, _I64, _I64, _P, _I32, _I64, _P, _P, _P, _I32,
                                       _I32, _P],
    "moeq_grouped_quantize_gather": [_I32, _P, _I64, _I64, _I64, _P, _I32, _I64, _P, _P, _I64,
                                     _P, _P, _P, _P, _I32, _I32, _I32, _P],
    "moeq_padded_scale_offsets": [_P, _P, _I32, _P],
    "moeq_grouped_matmul_rowwise_fp8": [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64,
                                        _I32, _I32, _I32, _P],
    "moeq_grouped_matmul_blockscaled": [_I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                        _I64, _I64, _I32, _I32, _I32, _P],
    "moeq_swiglu_quantize": [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I32, _I32, _P],
    "moeq_swiglu_quantize_mx": [_I32, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I32, _I32,
                                _P],
    "moeq_grouped_matmul_swiglu": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                   _I64, _I64, _I32, _I32, _I32, _P],
    "moeq_grouped_matmul_swiglu_mx": [_I32, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64,
                                      _I64, _I64, _I32, _I32, _I32, _P],
    "moeq_sf_swizzle": [_P, _P, _I64, _I64, _I64, _P],
    "moeq_sf_unswizzle": [_P, _P, _I64, _I64, _I64, _P],
    "moeq_interleave_gate_up": [_P, _P, _P, _I64, _I64, _I64, _P],
    "moeq_route_topk": [_P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _I32, _P],
    "moeq_quantize_topk": [_I32, _P, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P, _I32, _P, _P,
                           _I64, _P],
    "moeq_dispatch_scale_rows": [_I64, _I32, _I32, _I32],
    "moeq_grouped_amax_scale_topk": [_P, _I64, _I64, _I64, _P, _I32, _P, _I32, _P],
    "moeq_dispatch_mxfp4": [_P, _I64, _I64, _I64, _P, _I32, _I32, _P, _P, _I64, _P, _P, _P, _P,
                            _P, _I32, _P],
    "moeq_get_device_error": [_P, _U32P],
    "moeq_clear_device_error": [_P],
    "moeq_last_cuda_error": [],
    "moeq_status_string": [ctypes.c_int],
}
EXPORTS = tuple(_SIGNATURES)


class MoeqError(RuntimeError):
    def __init__(self, fn, status):
        code = lib().moeq_last_cuda_error() if status == 3 else 0
        super().__init__(f"{fn}: {STATUS.get(status, status)}" + (f" (cuda error {code})" if code else ""))
        self.status = status


def lib():
    """The loaded libmoeq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                               "python -m fp4_fp8_quantization_gb300.build")
        L = ctypes.CDLL(_LIB_PATH)
        for name, args in _SIGNATURES.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.moeq_status_string.restype = ctypes.c_char_p
        L.moeq_dispatch_scale_rows.restype = ctypes.c_int64
        _lib = L
    return _lib


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


def _ptr_rows(t, dtype, name):
    """Pointer of a 2-D tensor whose rows may be strided (unit element
    stride, row stride >= row length)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if t.dim() != 2 or t.stride(1) != 1 or t.stride(0) < t.shape[1]:
        raise ValueError(f"{name}: must be 2-D with unit column stride")
    return t.data_ptr()


def _call(fn, *args):
    st = getattr(lib(), fn)(*args)
    if st != 0:
        raise MoeqError(fn, st)


def _fmt(fmt):
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


_U8 = (torch.uint8, torch.float8_e4m3fn)
_U32 = (torch.uint32, torch.int32)


def grouped_amax_scale(inp, row_offsets, expert_ids, tensor_scale_out, num_experts,
                       num_active_experts=None, stream=None):
    G = expert_ids.numel() if num_active_experts is None else num_active_experts
    _call("moeq_grouped_amax_scale", _ptr_rows(inp, torch.bfloat16, "inp"), inp.stride(0),
          inp.shape[0], inp.shape[1], _ptr(row_offsets, _U32), _ptr(expert_ids, torch.int32),
          _ptr(tensor_scale_out, torch.float32), num_experts, G, _stream(stream))


def grouped_quantize(fmt, inp, out, scales, row_offsets, scales_offsets, expert_ids,
                     tensor_scale, num_experts, scale_rows_total, max_tokens_per_expert=0,
                     num_active_experts=None, stream=None):
    G = expert_ids.numel() if num_active_experts is None else num_active_experts
    _call("moeq_grouped_quantize", _fmt(fmt), _ptr_rows(inp, torch.bfloat16, "inp"), inp.stride(0),
          inp.shape[0], inp.shape[1], _ptr(out, _U8, "out"), _ptr(scales, _U8, "scales"),
          scale_rows_total, _ptr(row_offsets, _U32), _ptr(scales_offsets, _U32),
          _ptr(expert_ids, torch.int32), _ptr(tensor_scale, torch.float32), num_experts,
          max_tokens_per_expert, G, _stream(stream))


def grouped_amax_scale_gather(inp, indices, indices_divisor, row_offsets, expert_ids,
                              tensor_scale_out, num_experts, num_active_experts=None,
                              stream=None):
    G = expert_ids.numel() if num_active_experts is None else num_active_experts
    _call("moeq_grouped_amax_scale_gather", _ptr_rows(inp, torch.bfloat16, "inp"), inp.stride(0),
          inp.shape[0], inp.shape[1], _ptr(indices, torch.int32, "indices"), indices_divisor,
          indices.numel(), _ptr(row_offsets, _U32), _ptr(expert_ids, torch.int32),
          _ptr(tensor_scale_out, torch.float32), num_experts, G, _stream(stream))


def grouped_quantize_gather(fmt, inp, indices, indices_divisor, out, scales, row_offsets,
                            scales_offsets, expert_ids, tensor_scale, num_experts,
                            scale_rows_total, max_tokens_per_expert=0, num_active_experts=None,
                            stream=None):
    G = expert_ids.numel() if num_active_experts is None else num_active_experts
    _call("moeq_grouped_quantize_gather", _fmt(fmt), _ptr_rows(inp, torch.bfloat16, "inp"),
          inp.stride(0), inp.shape[0], inp.shape[1], _ptr(indices, torch.int32, "indices"),
          indices_divisor, indices.numel(), _ptr(out, _U8, "out"), _ptr(scales, _U8, "scales"),
          scale_rows_total, _ptr(row_offsets, _U32), _ptr(scales_offsets, _U32),
          _ptr(expert_ids, torch.int32), _ptr(tensor_scale, torch.float32), num_experts,
          max_tokens_per_expert, G, _stream(stream))


def padded_scale_offsets(row_offsets, scales_offsets, num_active_experts=None, stream=None):
    G = row_offsets.numel() - 1 if num_active_experts is None else num_active_experts
    _call("moeq_padded_scale_offsets", _ptr(row_offsets, _U32), _ptr(scales_offsets, _U32), G,
          _stream(stream))


def sf_swizzle(tiled, logical, stream=None):
    """logical uint8 [rows, kv] or [batch, rows, kv] -> the tiled block-scale
    layout in `tiled` (uint8, batch * sf_bytes(rows, kv) bytes)."""
    batch, rows, kv = (1, *logical.shape) if logical.dim() == 2 else logical.shape
    if tiled.numel() != batch * sf_bytes(rows, kv):
        raise ValueError("tiled: expected batch * sf_bytes(rows, kv) bytes")
    _call("moeq_sf_swizzle", _ptr(tiled, _U8, "tiled"), _ptr(logical, _U8, "logical"), batch,
          rows, kv, _stream(stream))


def sf_unswizzle(logical, tiled, stream=None):
    """The inverse of sf_swizzle: fills logical uint8 [rows, kv] or
    [batch, rows, kv] from the tiled buffer."""
    batch, rows, kv = (1, *logical.shape) if logical.dim() == 2 else logical.shape
    if tiled.numel() != batch * sf_bytes(rows, kv):
        raise ValueError("tiled: expected batch * sf_bytes(rows, kv) bytes")
    _call("moeq_sf_unswizzle", _ptr(logical, _U8, "logical"), _ptr(tiled, _U8, "tiled"), batch,
          rows, kv, _stream(stream))


def interleave_gate_up(out, gate, up, stream=None):
    """out[b, 2j] = gate[b, j], out[b, 2j + 1] = up[b, j]: uint8 gate, up
    [batch, rows, row_bytes] (or 2-D), out [batch, 2 * rows, row_bytes]."""
    if gate.shape != up.shape:
        raise ValueError("gate and up must have the same shape")
    batch, rows, rb = (1, *gate.shape) if gate.dim() == 2 else gate.shape
    if out.numel() != batch * 2 * rows * rb:
        raise ValueError("out: expected batch * 2 * rows * row_bytes bytes")
    _call("moeq_interleave_gate_up", _ptr(out, _U8, "out"), _ptr(gate, _U8, "gate"),
          _ptr(up, _U8, "up"), batch, rows, rb, _stream(stream))


def route_topk(topk_ids, row_offsets, expert_ids, src_info, scales_offsets=None, slot_rows=0,
               stream=None, dst_info=None):
    """Routes the choices of topk_ids (int32 [num_tokens, top_k]) to the
    groups of their experts: row_offsets (int32/uint32 [E + 1]), expert_ids
    (int32 [E]), src_info (int32 [num_tokens * top_k]) and, if given,
    scales_offsets ([E + 1]: padded, or slots of slot_rows rows) and
    dst_info (int32 [num_tokens * top_k], the row of each choice)."""
    if topk_ids.dim() != 2:
        raise ValueError("topk_ids: expected [num_tokens, top_k]")
    E = expert_ids.numel()
    if row_offsets.numel() != E + 1 or src_info.numel() < topk_ids.numel():
        raise ValueError("row_offsets [E + 1] and src_info [num_tokens * top_k] expected")
    _call("moeq_route_topk", _ptr(topk_ids, torch.int32, "topk_ids"), topk_ids.shape[0],
          topk_ids.shape[1], E, _ptr(row_offsets, _U32, "row_offsets"),
          _ptr(expert_ids, torch.int32, "expert_ids"), _ptr(src_info, torch.int32, "src_info"),
          _ptr(dst_info, torch.int32, "dst_info"), _ptr(scales_offsets, _U32, "scales_offsets"),
          slot_rows, _stream(stream))


def grouped_amax_scale_topk(tokens, topk_ids, tensor_scale_out, num_experts, stream=None):
    """Per-expert NVFP4 tensor scales from bf16 tokens [num_tokens, K] and
    their top-k expert ids (int32 [num_tokens, top_k]); each token read once."""
    if topk_ids.dim() != 2 or topk_ids.shape[0] != tokens.shape[0]:
        raise ValueError("topk_ids: expected [num_tokens, top_k]")
    _call("moeq_grouped_amax_scale_topk", _ptr_rows(tokens, torch.bfloat16, "tokens"),
          tokens.stride(0), tokens.shape[0], tokens.shape[1],
          _ptr(topk_ids, torch.int32, "topk_ids"), topk_ids.shape[1],
          _ptr(tensor_scale_out, torch.float32, "tensor_scale_out"), num_experts,
          _stream(stream))


def dispatch_scale_rows(num_tokens, top_k, num_experts, slot_rows=0):
    """Logical scale rows dispatch_mxfp4 needs for these sizes."""
    n = lib().moeq_dispatch_scale_rows(num_tokens, top_k, num_experts, slot_rows)
    if n < 0:
        raise ValueError("invalid sizes")
    return n


def quantize_topk(fmt, tokens, topk_ids, dst_info, out, scales, row_offsets, scales_offsets,
                  tensor_scale, num_experts, stream=None):
    """Token-major quantization of routed tokens (the bytes of
    grouped_quantize_gather on the routed rows, each token read once):
    tokens bf16 [num_tokens, K]; topk_ids int32 [num_tokens, top_k];
    dst_info, row_offsets, scales_offsets from route_topk; out
    [num_tokens * top_k, K / 2] (FP4) or [.., K] (MXFP8)."""
    if topk_ids.dim() != 2 or topk_ids.shape[0] != tokens.shape[0]:
        raise ValueError("topk_ids: expected [num_tokens, top_k]")
    T, K = tokens.shape
    v = 16 if fmt == "nvfp4" else 32
    rows = scales.numel() // max(1, sf_bytes(128, K // v)) * 128
    _call("moeq_quantize_topk", _fmt(fmt), _ptr_rows(tokens, torch.bfloat16, "tokens"),
          tokens.stride(0), T, K, _ptr(topk_ids, torch.int32, "topk_ids"), topk_ids.shape[1],
          _ptr(dst_info, torch.int32, "dst_info"), _ptr(row_offsets, _U32, "row_offsets"),
          _ptr(scales_offsets, _U32, "scales_offsets"),
          _ptr(tensor_scale, torch.float32, "tensor_scale"), num_experts,
          _ptr(out, _U8, "out"), _ptr(scales, _U8, "scales"), rows, _stream(stream))


def dispatch_mxfp4(tokens, topk_ids, out, scales, row_offsets, expert_ids, src_info,
                   scales_offsets, slot_rows=0, stream=None, dst_info=None):
    """Single-rank expert dispatch: route_topk, then MXFP4 quantization of
    the routed rows (row r is token src_info[r] // top_k).  tokens bf16
    [num_tokens, hidden]; out uint8 [num_tokens * top_k, hidden / 2]; scales
    the tiled E8M0 buffer (sf_bytes(rows, hidden / 32) bytes for
    rows = dispatch_scale_rows(...) or more, a multiple of 128)."""
    if topk_ids.dim() != 2 or topk_ids.shape[0] != tokens.shape[0]:
        raise ValueError("topk_ids: expected [num_tokens, top_k]")
    T, H = tokens.shape
    E = expert_ids.numel()
    if out.numel() < topk_ids.numel() * (H // 2) or row_offsets.numel() != E + 1:
        raise ValueError("out [num_tokens * top_k, hidden / 2] and row_offsets [E + 1] expected")
    rows = scales.numel() // max(1, sf_bytes(128, H // 32)) * 128
    if dst_info is None:   # the inverse routing map, device memory owned by the caller
        dst_info = torch.empty(topk_ids.numel(), dtype=torch.int32, device=tokens.device)
    _call("moeq_dispatch_mxfp4", _ptr_rows(tokens, torch.bfloat16, "tokens"), tokens.stride(0),
          T, H, _ptr(topk_ids, torch.int32, "topk_ids"), topk_ids.shape[1], E,
          _ptr(out, _U8, "out"), _ptr(scales, _U8, "scales"), rows,
          _ptr(row_offsets, _U32, "row_offsets"), _ptr(expert_ids, torch.int32, "expert_ids"),
          _ptr(src_info, torch.int32, "src_info"), _ptr(dst_info, torch.int32, "dst_info"),
          _ptr(scales_offsets, _U32, "scales_offsets"), slot_rows, _stream(stream))


def grouped_matmul_rowwise_fp8(c, a, b, a_scales, b_scales, a_offsets, expert_ids,
                               max_tokens_per_expert=0, num_active_experts=None, stream=None):
    G = expert_ids.numel() if num_active_experts is None else num_active_experts
    E, N, K = b.shape
    _call("moeq_grouped_matmul_rowwise_fp8", _ptr(c, torch.bfloat16, "c"), _ptr(a, _U8, "a"),
          _ptr(b, _U8, "b"), _ptr(a_scales, torch.float32), _ptr(b_scales, torch.float32),
          _ptr(a_offsets, _U32), _ptr(expert_ids, torch.int32), a.shape[0], N, K, E,
          max_tokens_per_expert, G, _stream(stream))


def grouped_matmul_blockscaled(fmt, c, a, a_sf, b, b_sf, expert_scales, a_offsets,
                               a_scales_offsets, expert_ids, N, K, scale_rows_total,
                               max_tokens_per_expert=0, num_active_experts=None, stream=None):
    G = expert_ids.numel() if num_active_experts is None else num_active_experts
    _call("moeq_grouped_matmul_blockscaled", _fmt(fmt), _ptr(c, torch.bfloat16, "c"),
          _ptr(a, _U8, "a"), _ptr(a_sf, _U8, "a_sf"), _ptr(b, _U8, "b"), _ptr(b_sf, _U8, "b_sf"),
          _ptr(expert_scales, torch.float32), _ptr(a_offsets, _U32), _ptr(a_scales_offsets, _U32),
          _ptr(expert_ids, torch.int32), a.shape[0], scale_rows_total, N, K, b.shape[0],
          max_tokens_per_expert, G, _stream(stream))


def swiglu_quantize(c_packed, c_sf, y, out_tensor_scale, a_offsets, a_scales_offsets,
                    expert_ids, num_experts, scale_rows_total, max_tokens_per_expert=0,
                    num_active_experts=None, stream=None):
    G = expert_ids.numel() if num_active_experts is None else num_active_experts
    _call("moeq_swiglu_quantize", _ptr(c_packed, _U8), _ptr(c_sf, _U8),
          _ptr(y, torch.bfloat16, "y"), _ptr(out_tensor_scale, torch.float32),
          _ptr(a_offsets, _U32), _ptr(a_scales_offsets, _U32), _ptr(expert_ids, torch.int32),
          y.shape[0], scale_rows_total, y.shape[1] // 2, num_experts, max_tokens_per_expert, G,
          _stream(stream))


def swiglu_quantize_mx(fmt, c_q, c_sf, y, a_offsets, a_scales_offsets, expert_ids, num_experts,
                       scale_rows_total, max_tokens_per_expert=0, num_active_experts=None,
                       stream=None):
    """Chained SwiGLU + MXFP4 / MXFP8 requantization (fmt "mxfp4" / "mxfp8")."""
    G = expert_ids.numel() if num_active_experts is None else num_active_experts
    _call("moeq_swiglu_quantize_mx", _fmt(fmt), _ptr(c_q, _U8), _ptr(c_sf, _U8),
          _ptr(y, torch.bfloat16, "y"), _ptr(a_offsets, _U32), _ptr(a_scales_offsets, _U32),
          _ptr(expert_ids, torch.int32), y.shape[0], scale_rows_total, y.shape[1] // 2,
          num_experts, max_tokens_per_expert, G, _stream(stream))


def grouped_matmul_swiglu(c_packed, c_sf, a, a_sf, b, b_sf, expert_scales, out_tensor_scale,
                          a_offsets, a_scales_offsets, expert_ids, I, K, scale_rows_total,
                          max_tokens_per_expert=0, num_active_experts=None, stream=None,
                          a_row_scales=None):
    G = expert_ids.numel() if num_active_experts is None else num_active_experts
    _call("moeq_grouped_matmul_swiglu", _ptr(c_packed, _U8), _ptr(c_sf, _U8), _ptr(a, _U8),
          _ptr(a_sf, _U8), _ptr(b, _U8), _ptr(b_sf, _U8), _ptr(expert_scales, torch.float32),
          _ptr(out_tensor_scale, torch.float32),
          _ptr(a_row_scales, torch.bfloat16, "a_row_scales"), _ptr(a_offsets, _U32),
          _ptr(a_scales_offsets, _U32), _ptr(expert_ids, torch.int32), a.shape[0],
          scale_rows_total, I, K, b.shape[0], max_tokens_per_expert, G, _stream(stream))


def grouped_matmul_swiglu_mx(fmt, c_q, c_sf, a, a_sf, b, b_sf, expert_scales, a_offsets,
                             a_scales_offsets, expert_ids, I, K, scale_rows_total,
                             max_tokens_per_expert=0, num_active_experts=None, stream=None):
    """Fused grouped MX matmul + SwiGLU + MX requantization (fmt "mxfp4" / "mxfp8")."""
    G = expert_ids.numel() if num_active_experts is None else num_active_experts
    _call("moeq_grouped_matmul_swiglu_mx", _fmt(fmt), _ptr(c_q, _U8), _ptr(c_sf, _U8),
          _ptr(a, _U8), _ptr(a_sf, _U8), _ptr(b, _U8), _ptr(b_sf, _U8),
          _ptr(expert_scales, torch.float32), _ptr(a_offsets, _U32),
          _ptr(a_scales_offsets, _U32), _ptr(expert_ids, torch.int32), a.shape[0],
          scale_rows_total, I, K, b.shape[0], max_tokens_per_expert, G, _stream(stream))


def get_device_error(stream=None):
    """Sticky device error bits (synchronises the stream)."""
    v = ctypes.c_uint32(0)
    st = lib().moeq_get_device_error(_stream(stream), ctypes.byref(v))
    if st not in (0, 4):
        raise MoeqError("moeq_get_device_error", st)
    return v.value


def clear_device_error(stream=None):
    _call("moeq_clear_device_error", _stream(stream))


def sf_bytes(rows, kv):
    """Bytes of a tiled block-scale buffer for [rows, kv] logical scales."""
    return (rows + 127) // 128 * ((kv + 3) // 4) * 512
