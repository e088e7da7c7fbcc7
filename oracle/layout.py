"""Block-scale memory layout (the index function), TEST INFRASTRUCTURE ONLY.

The pages give no layout: "max.nn.moe.NvMxf4f8Strategy" says only that the
activation scales are padded per expert (``grouped_quantize``) and that
``prepare_weight_scales`` rearranges the weight block scales into the
kernel's layout; "grouped_quantize_dynamic_scaled_fp4_async_kernel"
stores them through a TMA tile descriptor.  Reading adopted: the canonical
layout is the tensor core's tiled scale layout --

* logical scales are a [rows, Kv] byte matrix (Kv = K / block size);
* they are cut into atoms of 128 rows x 4 scale columns (512 bytes);
* inside an atom the byte of (row r, column c) sits at
  (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % 4);
* atoms are stored row-block-major: atom (rb, kb) starts at byte
  (rb * ceil(Kv / 4) + kb) * 512;
* bytes that belong to no logical scale (padding rows/columns) are 0.
"""
import numpy as np

ATOM_ROWS = 128
ATOM_COLS = 4
ATOM_BYTES = ATOM_ROWS * ATOM_COLS


def kv_atoms(kv):
    """Atom columns per 128-row block for Kv logical scale columns."""
    return (kv + ATOM_COLS - 1) // ATOM_COLS


def physical_bytes(rows, kv):
    """Size in bytes of the tiled buffer for [rows, kv] logical scales
    (rows rounded up to a whole number of 128-row atoms)."""
    rblocks = (rows + ATOM_ROWS - 1) // ATOM_ROWS
    return rblocks * kv_atoms(kv) * ATOM_BYTES


def sf_offset(r, c, kv):
    """Byte offset of logical scale (r, c) in the tiled buffer."""
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    atom = (r // ATOM_ROWS) * kv_atoms(kv) + c // ATOM_COLS
    inner = (r % 32) * 16 + ((r // 32) % 4) * 4 + (c % ATOM_COLS)
    return atom * ATOM_BYTES + inner


def swizzle(logical):
    """[rows, kv] logical scale bytes -> flat tiled buffer (padding = 0)."""
    logical = np.asarray(logical, dtype=np.uint8)
    rows, kv = logical.shape
    out = np.zeros(physical_bytes(rows, kv), dtype=np.uint8)
    rr, cc = np.meshgrid(np.arange(rows), np.arange(kv), indexing="ij")
    out[sf_offset(rr, cc, kv)] = logical
    return out


def unswizzle(buf, rows, kv):
    """Flat tiled buffer -> [rows, kv] logical scale bytes."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    rr, cc = np.meshgrid(np.arange(rows), np.arange(kv), indexing="ij")
    return buf[sf_offset(rr, cc, kv)]


def interleave_rows(gate, up):
    """Gate/up interleave of the fused SwiGLU weight ([..., rows, cols] ->
    [..., 2 rows, cols]): row 2j is gate row j, row 2j+1 is up row j.  The
    reading of "max.nn.moe.NvMxf4f8Strategy" adopted for the gate/up
    arrangement (granularity-1 interleave), applied to weight rows and to
    their logical block-scale rows alike."""
    gate = np.asarray(gate)
    up = np.asarray(up)
    assert gate.shape == up.shape
    out = np.empty(gate.shape[:-2] + (2 * gate.shape[-2], gate.shape[-1]), gate.dtype)
    out[..., 0::2, :] = gate
    out[..., 1::2, :] = up
    return out
