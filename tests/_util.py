"""Helpers shared by the GPU parity tests: ragged-group construction, the
GEMM tolerance, and host/device moves.  No quantization or GEMM arithmetic."""
import numpy as np
import pytest
import torch

from fp4_fp8_quantization_gb300 import synth

DEV = "cuda"


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def groups_from_counts(counts, expert_ids=None):
    """(a_offsets uint32 [G+1], expert_ids int32 [G]) for explicit counts."""
    counts = np.asarray(counts, np.int64)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    if expert_ids is None:
        expert_ids = np.arange(len(counts))
    return offs, np.asarray(expert_ids, np.int32)


def to_dev_u32(x):
    return torch.from_numpy(np.asarray(x, np.uint32).view(np.int32)).to(DEV)


def to_dev_i32(x):
    return torch.from_numpy(np.asarray(x, np.int32)).to(DEV)


def u8(t):
    """uint8 numpy view of a tensor (fp8 or uint8)."""
    t = t.detach().cpu()
    if t.dtype != torch.uint8:
        t = t.view(torch.uint8)
    return t.numpy()


def bf16_bits(t):
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_values(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


# Fields of the running test's metrics line (written by conftest.py when
# MOEQ_METRICS_LOG names a file).
NOTES = {}


def note(**fields):
    """Adds fields (sizes, error figures) to the running test's metrics line."""
    NOTES.update(fields)


def assert_gemm_close(gpu_bits, ref_f64, mask_rows=None):
    """Per element |gpu - ref| <= max(2 ulp_bf16(ref), 1e-3 * rms(ref)),
    ulp_bf16(x) = 2^(floor(log2|x|) - 7), rms over the compared elements."""
    got = bf16_values(gpu_bits).astype(np.float64)
    ref = np.asarray(ref_f64, np.float64)
    if mask_rows is not None:
        got, ref = got[mask_rows], ref[mask_rows]
    assert np.all(np.isfinite(ref)) and np.all(np.isfinite(got))
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 0.0
    with np.errstate(divide="ignore"):
        ulp = np.where(ref == 0, 0.0, 2.0 ** (np.floor(np.log2(np.abs(ref))) - 7))
    tol = np.maximum(2 * ulp, 1e-3 * rms)
    err = np.abs(got - ref)
    bad = err > tol
    if err.size:
        with np.errstate(divide="ignore", invalid="ignore"):
            ratio = np.where(err == 0, 0.0, err / tol)   # inf where tol is 0 and err is not
        note(compared=NOTES.get("compared", 0) + int(err.size),
             max_abs_err=max(NOTES.get("max_abs_err", 0.0), float(err.max())),
             max_err_over_tol=max(NOTES.get("max_err_over_tol", 0.0), float(ratio.max())))
    assert not bad.any(), (
        f"{bad.sum()} of {bad.size} outside tolerance; worst err {err.max():.4g} "
        f"(tol there {tol.reshape(-1)[np.argmax(err)]:.4g}), rms {rms:.4g}")


def sample_rows(a_offsets, n, seed=0):
    """n row indices spread over every non-empty group (first, last, random)."""
    rng = np.random.default_rng(seed)
    rows = set()
    for g in range(len(a_offsets) - 1):
        r0, r1 = int(a_offsets[g]), int(a_offsets[g + 1])
        if r1 > r0:
            rows.update({r0, r1 - 1})
    T = int(a_offsets[-1])
    rows.update(rng.integers(0, T, max(0, n - len(rows))).tolist())
    return np.array(sorted(rows), np.int64)


def group_sample_rows(a_offsets, block=128):
    """Per group (empty groups give an empty array): a row of its first
    `block`-row m-block, one of its middle m-block and its last row -- all
    rows of groups with at most 3."""
    out = []
    for g in range(len(a_offsets) - 1):
        r0, r1 = int(a_offsets[g]), int(a_offsets[g + 1])
        n = r1 - r0
        if n <= 3:
            out.append(np.arange(r0, r1, dtype=np.int64))
            continue
        nb = (n + block - 1) // block
        mb = nb // 2
        mid = r0 + mb * block + min(block // 2 + 5, n - 1 - mb * block)
        out.append(np.array(sorted({r0 + min(5, n - 1), mid, r1 - 1}), np.int64))
    return out


def tile_sample_cols(N, tile=256, offsets=(0, 1, 31, 32, 63, 64, 127, 128, 159, 200, 254, 255)):
    """Columns spread over every `tile`-wide n-tile of an N-column output
    (first and last columns of the tile and of its 32-column chunks)."""
    cols = {n0 + o for n0 in range(0, N, tile) for o in offsets if n0 + o < N}
    return np.array(sorted(cols), np.int64)


__all__ = ["synth"]
