"""Host-side bounds model of the grouped GEMM's copies and stores (CPU only).

The producer of `grouped_gemm_kernel` computes, per tile and k-step, the
coordinates of its TMA tensor loads and the byte ranges of its 1-D bulk
scale copies from the group offsets; the epilogue guards its global stores
by the group's row count.  This model restates that address arithmetic and
checks it on many ragged group layouts (empty groups, 1 / 127 / 128 / 129
rows, odd m-block counts in CTA pairs, N not a multiple of the tile):

* bulk copies (which have no out-of-bounds fill) stay inside their buffers;
* tensor loads start at an x that is a multiple of 16 bytes and at
  non-negative coordinates (loads past the end read zeros, by design);
* every stored output row and scale row lies in its buffer.
"""
import numpy as np
import pytest

ATOM = 512


def _groups(counts):
    ro = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    so = np.concatenate([[0], np.cumsum([(c + 127) // 128 * 128 for c in counts])]).astype(np.int64)
    return ro, so


def _check(counts, N, K, sf_vec, elem_bits, pair, bn=256, bm=128):
    """One launch's copies and stores; returns the number checked."""
    E = len(counts) + 2
    ids = np.random.default_rng(len(counts) + N).permutation(E)[:len(counts)]
    ro, so = _groups(counts)
    T = int(ro[-1])
    scale_rows_total = int(so[-1])
    kbytes = K * elem_bits // 8            # operand bytes per row
    kv_atoms = K // sf_vec // 4
    nrb = (N + 127) // 128
    RB = bn // 128
    KT = kbytes // 128
    sf_atoms = kv_atoms // KT
    a_sf_bytes = scale_rows_total // 128 * kv_atoms * ATOM
    b_sf_bytes = E * nrb * kv_atoms * ATOM
    NB = (N + bn - 1) // bn
    P = 2 if pair else 1
    checked = 0
    for g, rg in enumerate(counts):
        e = int(ids[g])
        mblocks = (rg + bm * P - 1) // (bm * P)          # tiles (pair tiles) of the group
        mlast = (rg + bm - 1) // bm - 1
        for tmb in range(mblocks):
            for nb in range(NB):
                n0 = nb * bn
                for rank in range(P):
                    mb = tmb * P + rank
                    row0 = int(ro[g]) + mb * bm
                    # A tensor load: x aligned, y >= 0 (past T reads zeros)
                    for kt in range(KT):
                        x = kt * 128
                        assert x % 16 == 0 and row0 >= 0
                    # B tensor load (each CTA of a pair its half of the rows)
                    assert n0 + rank * (bn // P) >= 0 and 0 <= e < E
                    # scale copies
                    sfa0 = (int(so[g]) // 128 + min(mb, mlast)) * kv_atoms
                    for kt in range(KT):
                        lo = (sfa0 + kt * sf_atoms) * ATOM
                        hi = lo + sf_atoms * ATOM
                        if pair:   # tensor copy of rows of 256 bytes: start row >= 0
                            assert lo >= 0
                        else:      # bulk copy: must lie in the buffer
                            assert 0 <= lo and hi <= a_sf_bytes, (g, mb, kt)
                        rbs = min(RB, nrb - n0 // 128)
                        for rb in range(RB if pair else rbs):
                            blk = e * nrb + n0 // 128 + rb
                            lo = (blk * kv_atoms + kt * sf_atoms) * ATOM
                            hi = lo + sf_atoms * ATOM
                            if pair:   # 3-D tensor copy; a block past the table reads zeros
                                assert blk >= 0
                            else:
                                assert 0 <= lo and hi <= b_sf_bytes, (g, rb, kt)
                    # epilogue stores: rows of the group only, scale rows of
                    # the group's padded range only
                    for lrow in range(mb * bm, mb * bm + bm):
                        if lrow < rg:
                            assert 0 <= int(ro[g]) + lrow < T
                        if mb * bm < rg:
                            assert int(so[g]) + lrow < int(so[g + 1]) <= scale_rows_total
                    checked += 1
    return checked


@pytest.mark.parametrize("kind,sf_vec,elem_bits,pair", [
    ("nvfp4", 16, 4, True), ("nvfp4", 16, 4, False), ("mxfp4", 32, 4, True),
    ("mxfp4", 32, 4, False), ("mxfp8", 32, 8, False)])
def test_blockscaled_copies_and_stores_in_bounds(kind, sf_vec, elem_bits, pair):
    rng = np.random.default_rng(5)
    layouts = [[0, 1, 127, 128, 129, 0, 300], [257], [1] * 9, [383, 0, 0, 129]]
    layouts += [list(rng.integers(0, 700, int(rng.integers(1, 12)))) for _ in range(20)]
    total = 0
    for counts in layouts:
        for N in (256, 384, 3072):
            total += _check(counts, N, 4096, sf_vec, elem_bits, pair,
                            bn=128 if kind == "mxfp8" else 256)
    assert total > 1000


def _staged_offset(row, piece):
    """Byte offset of 16-byte piece `piece` of row `row` in an epilogue warp's
    2 KB bf16 staging buffer: 64-byte rows, pieces XOR-swizzled by row pair."""
    return row * 64 + ((piece ^ ((row >> 1) & 3)) << 4)


@pytest.mark.parametrize("nvalid", [0, 1, 7, 8, 31, 32])
def test_staged_bf16_chunk_stores(nvalid):
    """The bf16 epilogue's staged stores of one 32 x 32 chunk: thread t
    writes its row t's four pieces, then in each of 4 rounds lane l reads
    row (l >> 2) + 8 i, piece l & 3 and stores it if the row is among the
    warp's first nvalid.  Every (valid row, piece) is stored exactly once, no
    other row, all offsets in the buffer, and each 8-lane phase of both
    passes touches 8 distinct groups of 4 banks (no bank conflict)."""
    stored = {}
    for i in range(4):
        for lane in range(32):
            row, piece = (lane >> 2) + 8 * i, lane & 3
            off = _staged_offset(row, piece)
            assert 0 <= off and off + 16 <= 2048
            if row < nvalid:
                stored[(row, piece)] = stored.get((row, piece), 0) + 1
    assert stored == {(r, k): 1 for r in range(nvalid) for k in range(4)}
    # the write pass: thread t stores piece j of its own row t
    for j in range(4):
        for phase in range(4):
            banks = {(_staged_offset(t, j) // 16) % 8 for t in range(8 * phase, 8 * phase + 8)}
            assert len(banks) == 8
    # the read pass
    for i in range(4):
        for phase in range(4):
            lanes = range(8 * phase, 8 * phase + 8)
            banks = {(_staged_offset((l >> 2) + 8 * i, l & 3) // 16) % 8 for l in lanes}
            assert len(banks) == 8
    # each written row's pieces are distinct 16-byte slots of that row
    for r in range(32):
        assert sorted(_staged_offset(r, k) - r * 64 for k in range(4)) == [0, 16, 32, 48]
