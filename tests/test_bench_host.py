"""Host-side arithmetic of bench.py's roofline block: the MMA floor of the
fused NVFP4 GEMM's own schedule (expert rows padded to 256-row CTA-pair
tiles of 256 columns, tiles dealt round-robin to the pairs, K / 64 MMAs of
128 cycles per tile)."""
import pytest

import bench
from fp4_fp8_quantization_gb300 import synth


def test_schedule_floor_counts_padded_pair_tiles():
    # rows 256 -> one pair tile, 257 -> two (the odd CTA of the second idle),
    # 0 -> none, 1 -> one; N = 512 -> two n-tiles: 8 pair tiles on 2 pairs
    ms, tiles, per_pair = bench.fp4_schedule_floor([256, 257, 0, 1], 512, 256, 4, 1000.0)
    assert (tiles, per_pair) == (8, 4)
    assert ms == pytest.approx(4 * (256 // 64) * 128 / 1e6)


def test_schedule_floor_ragged_n_and_uneven_deal():
    # N = 384 -> two n-tiles (the second half past N), one per pair
    ms, tiles, per_pair = bench.fp4_schedule_floor([100, 0, 0], 384, 4096, 4, 2000.0)
    assert (tiles, per_pair) == (2, 1)
    ms, tiles, per_pair = bench.fp4_schedule_floor([300], 256, 4096, 4, 2000.0)
    assert (tiles, per_pair) == (2, 1)
    # 600 rows -> 3 pair tiles on 2 pairs: the busiest runs 2
    ms, tiles, per_pair = bench.fp4_schedule_floor([600], 256, 4096, 4, 2000.0)
    assert (tiles, per_pair) == (3, 2)
    assert ms == pytest.approx(2 * 64 * 128 / 2e6)


def test_schedule_floor_of_the_128_expert_workload():
    # 16384 tokens top-8 over 128 experts: 62 experts above 1024 rows run a
    # fifth pair m-block, 6888 pair tiles instead of 6144, 91 on the busiest
    # of 76 pairs; 91 x 64 MMAs x 128 cycles at 2.07 GHz
    counts = synth.routing_counts(16384, 8, 128, seed=0)
    assert int((counts > 1024).sum()) == 62
    ms, tiles, per_pair = bench.fp4_schedule_floor(counts, 3072, 4096, 152, 2070.0)
    assert (tiles, per_pair) == (6888, 91)
    assert ms == pytest.approx(91 * 64 * 128 / 2.07e6)
